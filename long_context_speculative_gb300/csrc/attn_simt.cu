// CUDA-core verify attention: the split-KV history kernel for every dtype and
// head size (fp32 caches, d = 64, groups wider than the tensor-core kernel
// takes), and the merge kernel that adds the masked speculative part and
// combines all partials by log-sum-exp.
//
// Source of the decomposition: "LongSpec: Long-Context Lossless Speculative
// Decoding with Efficient Drafting and Verification", section 2.3 (Hybrid
// Tree Attention): unmasked attention over the history, masked attention over
// the speculative tokens, outputs merged with the log-sum-exp trick.
#include "attn.cuh"
#include "common.cuh"

namespace rapid {

namespace {

constexpr int kSimtThreads = 128;   // 4 warps
constexpr int kSimtRows = 64;       // group rows per CTA (16 per warp)
constexpr int kSimtRowsPerWarp = kSimtRows / 4;
constexpr int kSimtKeys = 32;       // key rows per smem tile (one per lane)

template <typename T>
struct Vec16;  // 16-byte vector of T
template <> struct Vec16<float> { static constexpr int N = 4; };
template <> struct Vec16<__nv_bfloat16> { static constexpr int N = 8; };

template <typename T>
__device__ __forceinline__ void load16_to_float(const T* src, float* dst);

template <>
__device__ __forceinline__ void load16_to_float<float>(const float* src, float* dst) {
    float4 v = *reinterpret_cast<const float4*>(src);
    dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
}

template <>
__device__ __forceinline__ void load16_to_float<__nv_bfloat16>(const __nv_bfloat16* src, float* dst) {
    uint4 v = *reinterpret_cast<const uint4*>(src);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        dst[2 * i] = __uint_as_float(w[i] << 16);
        dst[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// One CTA = (split s, block of up to 64 group rows, sequence b * Hkv + head g).
// Each lane owns one key of the 32-key tile for the scores and d/32 output
// columns for the PV product; scores live in the log2 domain.
template <typename T, int D>
__global__ void __launch_bounds__(kSimtThreads)
attn_prefix_simt_kernel(const AttnParams p) {
    constexpr int DP = D + 4;                 // padded K pitch: conflict-free float4 rows
    constexpr int NC = D / 32;                // output columns per lane
    constexpr int VN = Vec16<T>::N;
    extern __shared__ float4 smem_f4[];
    float* sQ = reinterpret_cast<float*>(smem_f4);   // [64][D], pre-scaled by scale*log2e
    float* sK = sQ + kSimtRows * D;                  // [32][DP]
    float* sV = sK + kSimtKeys * DP;                 // [32][D]

    griddep_wait();
    const int s = blockIdx.x;
    const int rb = blockIdx.y;
    const int bg = blockIdx.z;
    const int b = bg / p.Hkv;
    const int g = bg % p.Hkv;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int r0 = rb * kSimtRows;
    const int nrows = min(kSimtRows, p.R - r0);

    const int64_t P = clamped_prefix(p, b);
    const int64_t lo = (int64_t)s * p.chunk;
    const int64_t hi = (lo + p.chunk < P) ? lo + p.chunk : P;

    const T* Qg = static_cast<const T*>(p.Q) + ((int64_t)b * p.Hq + (int64_t)g * p.G) * p.n_q * D;
    for (int idx = threadIdx.x; idx < kSimtRows * D; idx += kSimtThreads) {
        const int r = idx / D;
        const int k = idx - r * D;
        sQ[idx] = (r < nrows) ? to_float(Qg[(int64_t)(r0 + r) * D + k]) * p.scale_log2 : 0.f;
    }

    float acc[kSimtRowsPerWarp][NC];
    float m[kSimtRowsPerWarp], l[kSimtRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kSimtRowsPerWarp; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[i][c] = 0.f;
    }

    const T* Kh = static_cast<const T*>(p.K) + (int64_t)bg * p.cap * D;
    const T* Vh = static_cast<const T*>(p.V) + (int64_t)bg * p.cap * D;

    for (int64_t t0 = lo; t0 < hi; t0 += kSimtKeys) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < kSimtKeys * (D / VN); idx += kSimtThreads) {
            const int key = idx / (D / VN);
            const int k = (idx - key * (D / VN)) * VN;
            float tk[VN], tv[VN];
            if (t0 + key < hi) {
                load16_to_float<T>(Kh + (t0 + key) * D + k, tk);
                load16_to_float<T>(Vh + (t0 + key) * D + k, tv);
            } else {
#pragma unroll
                for (int e = 0; e < VN; ++e) { tk[e] = 0.f; tv[e] = 0.f; }
            }
#pragma unroll
            for (int e = 0; e < VN; ++e) {
                sK[key * DP + k + e] = tk[e];
                sV[key * D + k + e] = tv[e];
            }
        }
        __syncthreads();

        const bool valid = (t0 + lane) < hi;
        float sc[kSimtRowsPerWarp];
#pragma unroll
        for (int i = 0; i < kSimtRowsPerWarp; ++i) sc[i] = 0.f;
#pragma unroll 4
        for (int k = 0; k < D; k += 4) {
            const float4 kv = *reinterpret_cast<const float4*>(&sK[lane * DP + k]);
#pragma unroll
            for (int i = 0; i < kSimtRowsPerWarp; ++i) {
                const int r = warp + 4 * i;
                if (r < nrows) {
                    const float4 qv = *reinterpret_cast<const float4*>(&sQ[r * D + k]);
                    sc[i] = fmaf(qv.x, kv.x, sc[i]);
                    sc[i] = fmaf(qv.y, kv.y, sc[i]);
                    sc[i] = fmaf(qv.z, kv.z, sc[i]);
                    sc[i] = fmaf(qv.w, kv.w, sc[i]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kSimtRowsPerWarp; ++i) {
            if (warp + 4 * i >= nrows) continue;
            const float si = valid ? sc[i] : -INFINITY;
            const float mnew = fmaxf(m[i], warp_max(si));
            const float corr = exp2f(m[i] - mnew);
            const float pj = exp2f(si - mnew);
            l[i] = l[i] * corr + warp_sum(pj);
            m[i] = mnew;
#pragma unroll
            for (int c = 0; c < NC; ++c) acc[i][c] *= corr;
            sc[i] = pj;
        }
        const int nk = (hi - t0 < kSimtKeys) ? (int)(hi - t0) : kSimtKeys;
        for (int j = 0; j < nk; ++j) {
            float vv[NC];
#pragma unroll
            for (int c = 0; c < NC; ++c) vv[c] = sV[j * D + lane + 32 * c];
#pragma unroll
            for (int i = 0; i < kSimtRowsPerWarp; ++i) {
                const float pj = __shfl_sync(0xffffffffu, sc[i], j);
#pragma unroll
                for (int c = 0; c < NC; ++c) acc[i][c] = fmaf(pj, vv[c], acc[i][c]);
            }
        }
    }

    // Partial of this split: acc, (m, l).  An empty split leaves m = -inf, l = 0.
    const int64_t slot = ((int64_t)bg * p.nparts + s) * p.R;
#pragma unroll
    for (int i = 0; i < kSimtRowsPerWarp; ++i) {
        const int r = warp + 4 * i;
        if (r >= nrows) continue;
        float* dst = p.part_acc + (slot + r0 + r) * D;
#pragma unroll
        for (int c = 0; c < NC; ++c) dst[lane + 32 * c] = acc[i][c];
        if (lane == 0) {
            p.part_ml[(slot + r0 + r) * 2 + 0] = m[i];
            p.part_ml[(slot + r0 + r) * 2 + 1] = l[i];
        }
    }
}

// One CTA of 128 threads per query row (b, h, i): the log-sum-exp merge of
// the history partials (and, when the history kernel did not cover them, the
// masked attention over the n_q speculative rows):
//   M = max(m_spec, m_s);  L = sum_parts l_part 2^(m_part - M);
//   O = sum_parts acc_part 2^(m_part - M) / L;   LSE = (M + log2 L) ln 2.
// Warps split the partials (s = warp, warp + 4, ...), lanes split the d
// columns, so every load of a partial row is independent of the others.
constexpr int kMergeThreads = 128;
constexpr int kMergeMaxS = 1024;

template <typename T, int D>
__global__ void __launch_bounds__(kMergeThreads) attn_merge_kernel(const AttnParams p) {
    constexpr int VPL = D / 32;                 // columns per lane
    __shared__ float s_w[kMergeMaxS];           // partial weights 2^(m_s - M)
    __shared__ float2 s_ml[kMergeMaxS];         // (m_s, l_s) of the partials
    __shared__ float s_red[4][D];
    __shared__ float s_scal[4][2];
    __shared__ float s_spec[2];                 // m_spec, l_spec (relative to m_spec)
    griddep_wait();
    griddep_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = blockIdx.x;
    const int bg = blockIdx.y;
    const int b = bg / p.Hkv;
    const int g = bg % p.Hkv;
    const int h = g * p.G + r / p.n_q;
    const int i = r % p.n_q;
    // A device-side input the host cannot check: once per sequence, a history
    // length outside [0, kv_capacity - n_q] (clamped everywhere) sets the
    // bad-input bit of the error word.  (A mask row may hide every
    // speculative row, even the query's own node: a key-range shard of the
    // history that must not see them passes an all-zero mask.)
    if (tid == 0 && g == 0 && r == 0 && p.err) {
        const int64_t P = p.prefix_len[b];
        if (P < 0 || P > p.cap - p.n_q) atomicOr(p.err, kErrBadInput);
    }
    // partial slots written for this sequence: all S of (b, g) for the
    // CUDA-core history kernel; the S_b slots from part_first for the
    // tensor-core kernel
    const int nparts = p.balanced ? p.part_nsplit[bg] : p.nparts;
    const int64_t first = p.balanced ? (int64_t)g * p.nparts + p.part_first[bg]
                                     : (int64_t)bg * p.nparts;
    const float* ml = p.part_ml + (first * p.R + r) * 2;     // + s * R * 2
    const float* pa = p.part_acc + (first * p.R + r) * D;    // + s * R * D
    const int64_t mls = (int64_t)p.R * 2, pas = (int64_t)p.R * D;

    // ---- speculative rows (warp 0), only when the history kernel skipped them
    float acc_spec[VPL];
#pragma unroll
    for (int c = 0; c < VPL; ++c) acc_spec[c] = 0.f;
    float m_spec = -INFINITY;
    if (warp == 0) {
        float l_spec = 0.f;
        if (!p.spec_in_partials) {
            const int64_t P = clamped_prefix(p, b);
            const T* Qrow = static_cast<const T*>(p.Q) + (((int64_t)b * p.Hq + h) * p.n_q + i) * D;
            const T* Kh = static_cast<const T*>(p.K) + (int64_t)bg * p.cap * D;
            const T* Vh = static_cast<const T*>(p.V) + (int64_t)bg * p.cap * D;
            float q[VPL];
#pragma unroll
            for (int c = 0; c < VPL; ++c) q[c] = to_float(Qrow[lane * VPL + c]) * p.scale_log2;
            for (int j = 0; j < p.n_q; ++j) {
                const bool vis =
                    p.mask ? (p.mask[((int64_t)b * p.n_q + i) * p.n_q + j] != 0) : (j <= i);
                if (!vis) continue;                                   // warp-uniform
                const T* kr = Kh + (P + j) * D + lane * VPL;
                const T* vr = Vh + (P + j) * D + lane * VPL;
                float dot = 0.f;
#pragma unroll
                for (int c = 0; c < VPL; ++c) dot = fmaf(q[c], to_float(kr[c]), dot);
                const float sj = warp_sum(dot);
                const float mnew = fmaxf(m_spec, sj);
                const float corr = exp2f(m_spec - mnew);
                const float pj = exp2f(sj - mnew);
                l_spec = l_spec * corr + pj;
#pragma unroll
                for (int c = 0; c < VPL; ++c) acc_spec[c] = fmaf(pj, to_float(vr[c]), acc_spec[c] * corr);
                m_spec = mnew;
            }
        }
        if (lane == 0) { s_spec[0] = m_spec; s_spec[1] = l_spec; }
    }
    // ---- the first partial rows into registers at once (warp w takes the
    // partials w, w + 4, ...), while the (m, l) pairs are reduced: one round of
    // memory latency instead of three
    constexpr int kPre = 8;                      // partial rows per warp held in registers
    float v[kPre][VPL];
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
        const int sp = warp + 4 * u;
#pragma unroll
        for (int c = 0; c < VPL; ++c) v[u][c] = sp < nparts ? pa[sp * pas + lane * VPL + c] : 0.f;
    }
    // ---- M over the history partials -------------------------------------
    float mloc = -INFINITY;
    for (int s = tid; s < nparts; s += kMergeThreads) {
        const float2 x = *reinterpret_cast<const float2*>(ml + s * mls);
        s_ml[s] = x;
        if (x.y > 0.f) mloc = fmaxf(mloc, x.x);
    }
    mloc = warp_max(mloc);
    if (lane == 0) s_scal[warp][0] = mloc;
    __syncthreads();
    const float M = fmaxf(fmaxf(fmaxf(s_scal[0][0], s_scal[1][0]), fmaxf(s_scal[2][0], s_scal[3][0])),
                          s_spec[0]);
    // ---- weights and L ---------------------------------------------------
    float lloc = 0.f;
    for (int s = tid; s < nparts; s += kMergeThreads) {
        const float2 x = s_ml[s];
        const float w = x.y > 0.f ? exp2f(x.x - M) : 0.f;
        s_w[s] = w;
        lloc = fmaf(w, x.y, lloc);
    }
    lloc = warp_sum(lloc);
    if (lane == 0) s_scal[warp][1] = lloc;
    __syncthreads();
    const float wspec = (s_spec[1] > 0.f) ? exp2f(s_spec[0] - M) : 0.f;
    const float L = (s_scal[0][1] + s_scal[1][1]) + (s_scal[2][1] + s_scal[3][1]) + wspec * s_spec[1];
    // ---- weighted partial rows ---------------------------------------------
    float acc[VPL];
#pragma unroll
    for (int c = 0; c < VPL; ++c) acc[c] = 0.f;
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
        const int sp = warp + 4 * u;
        const float w = sp < nparts ? s_w[sp] : 0.f;
#pragma unroll
        for (int c = 0; c < VPL; ++c) acc[c] = fmaf(w, w != 0.f ? v[u][c] : 0.f, acc[c]);
    }
    for (int s = warp + 4 * kPre; s < nparts; s += 4) {
        const float w = s_w[s];
        if (w == 0.f) continue;
#pragma unroll
        for (int c = 0; c < VPL; ++c) acc[c] = fmaf(w, pa[s * pas + lane * VPL + c], acc[c]);
    }
#pragma unroll
    for (int c = 0; c < VPL; ++c) s_red[warp][lane * VPL + c] = acc[c];
    __syncthreads();
    if (warp == 0) {
        T* Orow = static_cast<T*>(p.O) + (((int64_t)b * p.Hq + h) * p.n_q + i) * D;
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int c = 0; c < VPL; ++c) {
            const int col = lane * VPL + c;
            const float o = (s_red[0][col] + s_red[1][col]) + (s_red[2][col] + s_red[3][col]) +
                            wspec * acc_spec[c];
            Orow[col] = from_float<T>(o * inv);
        }
        if (lane == 0)
            p.LSE[((int64_t)b * p.Hq + h) * p.n_q + i] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
}

template <typename T, int D>
cudaError_t launch_simt_typed(const AttnParams& p, cudaStream_t st) {
    const int smem = (kSimtRows * D + kSimtKeys * (D + 4) + kSimtKeys * D) * (int)sizeof(float);
    auto kern = attn_prefix_simt_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.S, (p.R + kSimtRows - 1) / kSimtRows, p.B * p.Hkv);
    kern<<<grid, kSimtThreads, smem, st>>>(p);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_merge_typed(const AttnParams& p, cudaStream_t st) {
    // partials per row: at most nparts for the CUDA-core kernel; S_b <=
    // nparts - B + 1 for the tensor-core kernel (every sequence has a split)
    if ((p.balanced ? p.nparts - p.B + 1 : p.nparts) > kMergeMaxS) return cudaErrorNotSupported;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.R, p.B * p.Hkv, 1);
    cfg.blockDim = dim3(kMergeThreads, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_merge_kernel<T, D>, p);
}

}  // namespace

cudaError_t launch_attn_prefix_simt(const AttnParams& p, int dtype, cudaStream_t s) {
    if (dtype == 1) {
        return p.d == 128 ? launch_simt_typed<__nv_bfloat16, 128>(p, s)
                          : launch_simt_typed<__nv_bfloat16, 64>(p, s);
    }
    return p.d == 128 ? launch_simt_typed<float, 128>(p, s) : launch_simt_typed<float, 64>(p, s);
}

cudaError_t launch_attn_merge(const AttnParams& p, int dtype, cudaStream_t s) {
    if (dtype == 1) {
        return p.d == 128 ? launch_merge_typed<__nv_bfloat16, 128>(p, s)
                          : launch_merge_typed<__nv_bfloat16, 64>(p, s);
    }
    return p.d == 128 ? launch_merge_typed<float, 128>(p, s) : launch_merge_typed<float, 64>(p, s);
}

}  // namespace rapid
