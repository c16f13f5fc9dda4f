// Retrieval-augmented acceptance over the full vocabulary.
//
// Source: "RAPID: Long-Context Inference with Retrieval-Augmented Speculative
// Decoding" (blog summary).  Section 2.1: accept a draft x' iff
// r <= min(1, p(x')/q(x')), r ~ U(0,1); on rejection draw from the residual
// norm(max(p - q, 0)).  Section 2.4: p = softmax(z/T), the
// retrieval-augmented target p_hat = softmax(z/T + eta (q - p)) (Eq. 4),
// entries of p_hat below 0.1 * max p_hat replaced by those of p, p_hat used in
// the ratio test, and the adjusted residual norm(max(p - p_hat, p - q)).
//
// Layout of the work: one thread-block cluster per vocabulary row (b, j); the
// row is cut into `chunk`-sized pieces, one per CTA, bulk-copied (TMA) into
// shared memory.  Three vocabulary-wide reductions (the softmax of z/T, the
// softmax of the augmented logits, the residual mass) combine across the
// cluster through distributed shared memory.  Every row settles the ratio test
// of each draft node scored by it and draws its one candidate next token
// (uniform u_{j+1}): the adjusted residual if the row has children, else the
// bonus draw from p.  A second small kernel walks the chain or tree and picks
// n_accepted and the next token from those per-row results.
#include <cooperative_groups.h>

#include "accept.cuh"
#include "common.cuh"

namespace cg = cooperative_groups;

namespace rapid {

namespace {

constexpr int kNT = kAcceptThreads;
constexpr int kWarps = kNT / 32;

struct MS {
    float m, s;
};

// (m_a, s_a) + (m_b, s_b) for sums of exp(x - m): rescale to the larger max.
__device__ __forceinline__ MS ms_combine(MS a, MS b) {
    const float m = fmaxf(a.m, b.m);
    if (m == -INFINITY) return MS{-INFINITY, 0.f};
    const float sa = a.s > 0.f ? a.s * exp2f((a.m - m) * kLog2e) : 0.f;
    const float sb = b.s > 0.f ? b.s * exp2f((b.m - m) * kLog2e) : 0.f;
    return MS{m, sa + sb};
}

__device__ __forceinline__ MS warp_ms(MS v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        MS w;
        w.m = __shfl_xor_sync(0xffffffffu, v.m, o);
        w.s = __shfl_xor_sync(0xffffffffu, v.s, o);
        v = ms_combine(v, w);
    }
    return v;
}

struct RowShared {
    uint64_t bar;
    int n_children;
    int children[kAcceptMaxNq];
    MS red_ms[kWarps];
    float red_f[kWarps][16];
    float stripe_total[16];
    float warp_tot[kWarps];
    // cluster exchange slots (read by peers through distributed shared memory)
    MS x_ms1;
    MS x_ms2;
    float x_w;
    int pick_thread;
    int last_thread;
};

__device__ __forceinline__ int parent_of(const AcceptParams& p, int b, int i) {
    if (!p.parent) return i - 1;
    int par = p.parent[(int64_t)b * p.n_q + i];
    if (par < 0) par = 0;
    if (par > i - 1) par = i - 1;
    return par;
}

// Block-wide (m, s) combine; result valid in every thread.
__device__ MS block_ms(MS v, RowShared& sh) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    v = warp_ms(v);
    __syncthreads();
    if (lane == 0) sh.red_ms[warp] = v;
    __syncthreads();
    MS acc = sh.red_ms[0];
    for (int w = 1; w < kWarps; ++w) acc = ms_combine(acc, sh.red_ms[w]);
    return acc;
}

template <int F>
__global__ void __launch_bounds__(kNT)
accept_rows_kernel(const AcceptParams p) {
    constexpr int E = 4 * F;
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int row = blockIdx.y;                 // b * n_q + j
    const int b = row / p.n_q;
    const int j = row - b * p.n_q;
    const int t = threadIdx.x;

    extern __shared__ float4 dyn_f4[];
    float* sz = reinterpret_cast<float*>(dyn_f4);
    float* sq = sz + p.chunk;
    __shared__ RowShared sh;
    griddep_wait();

    const int64_t lo = (int64_t)rank * p.chunk;
    int64_t n64 = (int64_t)p.V - lo;
    if (n64 > p.chunk) n64 = p.chunk;
    if (n64 < 0) n64 = 0;
    const int n = (int)n64;
    const float* zrow = p.z + (int64_t)row * p.V + lo;
    const float* qrow = p.q + (int64_t)row * p.V + lo;

    // ---- stage this CTA's piece of z and q in shared memory -------------
    if (p.bulk) {
        if (t == 0) {
            mbar_init(&sh.bar, 1);
            fence_mbar_init();
        }
        __syncthreads();
        if (t == 0) {
            mbar_arrive_expect_tx(&sh.bar, (uint32_t)(n * 8));
            if (n > 0) {
                bulk_g2s(sz, zrow, (uint32_t)(n * 4), &sh.bar);
                bulk_g2s(sq, qrow, (uint32_t)(n * 4), &sh.bar);
            }
        }
    } else {
        for (int e = t; e < n; e += kNT) {
            sz[e] = zrow[e];
            sq[e] = qrow[e];
        }
    }
    // children of row j (nodes scored by this row)
    if (t == 0) {
        int nc = 0;
        for (int c = j + 1; c < p.n_q; ++c)
            if (parent_of(p, b, c) == j) sh.children[nc++] = c;
        sh.n_children = nc;
    }
    if (p.bulk) mbar_wait(&sh.bar, 0, p.err);
    __syncthreads();
    const bool has_children = sh.n_children > 0;

    // ---- pass 1: p = softmax(z / T) -----------------------------------
    float xr[E], er[E];
    float m_t = -INFINITY;
#pragma unroll
    for (int f = 0; f < F; ++f) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int el = 4 * (t + f * kNT) + c;
            const float x = el < n ? sz[el] * p.invT : -INFINITY;
            xr[4 * f + c] = x;
            m_t = fmaxf(m_t, x);
        }
    }
    float s_t = 0.f;
#pragma unroll
    for (int k = 0; k < E; ++k) {
        er[k] = (xr[k] == -INFINITY) ? 0.f : exp2f((xr[k] - m_t) * kLog2e);
        s_t += er[k];
    }
    MS cta1 = block_ms(MS{m_t, s_t}, sh);
    if (t == 0) sh.x_ms1 = cta1;
    cluster.sync();
    MS tot1 = MS{-INFINITY, 0.f};
    for (int c = 0; c < C; ++c) tot1 = ms_combine(tot1, cluster.map_shared_rank(&sh, c)->x_ms1);
    // p_k = er_k * f_t
    const float f_t = (m_t == -INFINITY) ? 0.f : exp2f((m_t - tot1.m) * kLog2e) / tot1.s;

    // ---- pass 2: p_hat = softmax(z/T + eta (q - p)) ----------------------
    float m2_t = -INFINITY;
#pragma unroll
    for (int f = 0; f < F; ++f) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int k = 4 * f + c;
            const int el = 4 * (t + f * kNT) + c;
            if (el < n) {
                const float pk = er[k] * f_t;
                xr[k] = xr[k] + p.eta * (sq[el] - pk);
            }
            m2_t = fmaxf(m2_t, xr[k]);
        }
    }
    float s2_t = 0.f;
#pragma unroll
    for (int k = 0; k < E; ++k) {
        xr[k] = (xr[k] == -INFINITY) ? 0.f : exp2f((xr[k] - m2_t) * kLog2e);
        s2_t += xr[k];
    }
    MS cta2 = block_ms(MS{m2_t, s2_t}, sh);
    if (t == 0) sh.x_ms2 = cta2;
    cluster.sync();
    MS tot2 = MS{-INFINITY, 0.f};
    for (int c = 0; c < C; ++c) tot2 = ms_combine(tot2, cluster.map_shared_rank(&sh, c)->x_ms2);
    // p_hat_k = xr_k * g_t; max_k p_hat_k = 1 / s2 (the arg-max term is exp(0)).
    const float g_t = (m2_t == -INFINITY) ? 0.f : exp2f((m2_t - tot2.m) * kLog2e) / tot2.s;
    const float thr = p.clamp ? 0.1f * (1.0f / tot2.s) : -1.0f;

    // ---- ratio test of every draft node scored by this row -------------
    for (int ci = 0; ci < sh.n_children; ++ci) {
        const int node = sh.children[ci];
        const int tok = p.tokens[(int64_t)b * p.n_q + node];
        const int64_t el = (int64_t)tok - lo;
        if (tok < 0 || tok >= p.V || el < 0 || el >= n) continue;   // owner only
        const int e4 = (int)el >> 2;
        if ((e4 % kNT) != t) continue;
        const int kk = 4 * (e4 / kNT) + ((int)el & 3);
        float ek = 0.f, hk = 0.f;
#pragma unroll
        for (int k = 0; k < E; ++k)
            if (k == kk) { ek = er[k]; hk = xr[k]; }
        const float pt = ek * f_t;
        float ph = hk * g_t;
        if (ph < thr) ph = pt;
        const float qt = sq[el];
        const float ratio = (qt == 0.f) ? INFINITY : ph / qt;
        const Philox4 rnd = philox4x32_10((uint32_t)node, (uint32_t)b, 0u, 0u, p.seed_lo, p.seed_hi);
        const float r = word_uniform(rnd.w[0]);
        p.ws_accept[(int64_t)b * p.n_q + node] = (r <= fminf(1.0f, ratio)) ? 1 : 0;
        if (p.diag) {
            float* dg = p.diag + ((int64_t)b * p.n_q + node) * 5;
            dg[0] = pt; dg[1] = ph; dg[2] = qt; dg[3] = ratio; dg[4] = r;
        }
    }
    // Out-of-range draft tokens are rejected (memory-safe handling of bad input).
    if (rank == 0 && t == 0) {
        for (int ci = 0; ci < sh.n_children; ++ci) {
            const int node = sh.children[ci];
            const int tok = p.tokens[(int64_t)b * p.n_q + node];
            if (tok < 0 || tok >= p.V) p.ws_accept[(int64_t)b * p.n_q + node] = 0;
        }
    }

    if (t == 0) griddep_launch_dependents();

    // ---- pass 3: candidate next token of this row ------------------------
    const Philox4 rnd = philox4x32_10((uint32_t)(j + 1), (uint32_t)b, 0u, 0u, p.seed_lo, p.seed_hi);
    const float u = word_uniform(rnd.w[1]);
    bool residual = has_children;
    for (int attempt = 0; attempt < 2; ++attempt) {
        float wsum[F];
#pragma unroll
        for (int f = 0; f < F; ++f) {
            float acc = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int k = 4 * f + c;
                const int el = 4 * (t + f * kNT) + c;
                float w = 0.f;
                if (el < n) {
                    const float pk = er[k] * f_t;
                    if (residual) {
                        float ph = xr[k] * g_t;
                        if (ph < thr) ph = pk;
                        w = fmaxf(fmaxf(pk - ph, pk - sq[el]), 0.f);
                    } else {
                        w = pk;
                    }
                }
                acc += w;
            }
            wsum[f] = acc;
        }
        // stripe totals (stripe f = the f-th run of kNT float4s of this CTA)
        const int warp = t >> 5, lane = t & 31;
#pragma unroll
        for (int f = 0; f < F; ++f) {
            const float v = warp_sum(wsum[f]);
            if (lane == 0) sh.red_f[warp][f] = v;
        }
        __syncthreads();
        if (t < F) {
            float s = 0.f;
            for (int w = 0; w < kWarps; ++w) s += sh.red_f[w][t];
            sh.stripe_total[t] = s;
        }
        __syncthreads();
        float Wc = 0.f;
        for (int f = 0; f < F; ++f) Wc += sh.stripe_total[f];
        if (t == 0) sh.x_w = Wc;
        cluster.sync();
        float W = 0.f;
        for (int c = 0; c < C; ++c) W += cluster.map_shared_rank(&sh, c)->x_w;
        if (residual && !(W > 0.f)) {   // residual without mass: fall back to p
            residual = false;
            cluster.sync();             // peers done reading x_w before it is rewritten
            continue;
        }

        // CTA level: first CTA whose running total passes u*W (else the last
        // CTA with mass), and the target inside it.
        const float target = u * W;
        int owner = -1, last_pos = -1;
        float cum = 0.f, t_in = INFINITY;
        for (int c = 0; c < C; ++c) {
            const float wc = cluster.map_shared_rank(&sh, c)->x_w;
            if (wc > 0.f) {
                last_pos = c;
                if (owner < 0 && cum + wc > target) { owner = c; t_in = target - cum; }
            }
            cum += wc;
        }
        if (owner < 0) { owner = last_pos; t_in = INFINITY; }
        if (owner == rank) {
            // stripe level
            int fs = -1, flast = -1;
            float cs = 0.f, t_s = INFINITY;
            for (int f = 0; f < F; ++f) {
                const float v = sh.stripe_total[f];
                if (v > 0.f) {
                    flast = f;
                    if (fs < 0 && cs + v > t_in) { fs = f; t_s = t_in - cs; }
                }
                cs += v;
            }
            if (fs < 0) { fs = flast; t_s = INFINITY; }
            // thread level: exclusive scan of this stripe's per-thread sums
            float v = 0.f;
#pragma unroll
            for (int f = 0; f < F; ++f)
                if (f == fs) v = wsum[f];
            float incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane == 31) sh.warp_tot[warp] = incl;
            if (t == 0) { sh.pick_thread = kNT; sh.last_thread = -1; }
            __syncthreads();
            float woff = 0.f;
            for (int w = 0; w < warp; ++w) woff += sh.warp_tot[w];
            float excl = __shfl_up_sync(0xffffffffu, incl, 1);
            if (lane == 0) excl = 0.f;
            excl += woff;
            if (v > 0.f) {
                atomicMax(&sh.last_thread, t);
                if (excl + v > t_s) atomicMin(&sh.pick_thread, t);
            }
            __syncthreads();
            int pick = sh.pick_thread;
            const bool fallback = (pick >= kNT);
            if (fallback) pick = sh.last_thread;
            if (t == pick && fs >= 0) {
                // element level inside this thread's float4 of stripe fs
                int kpick = -1, klast = -1;
                float ce = excl;
                const float t_e = fallback ? INFINITY : t_s;
#pragma unroll
                for (int f = 0; f < F; ++f) {
                    if (f != fs) continue;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int k = 4 * f + c;
                        const int el = 4 * (t + f * kNT) + c;
                        float w = 0.f;
                        if (el < n) {
                            const float pk = er[k] * f_t;
                            if (residual) {
                                float ph = xr[k] * g_t;
                                if (ph < thr) ph = pk;
                                w = fmaxf(fmaxf(pk - ph, pk - sq[el]), 0.f);
                            } else {
                                w = pk;
                            }
                        }
                        if (w > 0.f) {
                            klast = c;
                            if (kpick < 0 && ce + w > t_e) kpick = c;
                        }
                        ce += w;
                    }
                }
                if (kpick < 0) kpick = klast;
                if (kpick < 0) kpick = 0;   // unreachable: the stripe has mass
                p.ws_sample[row] = (int)(lo + 4 * (t + fs * kNT) + kpick);
            }
            if (t == 0 && (pick < 0 || fs < 0)) p.ws_sample[row] = (int)lo;   // unreachable guard
        }
        break;
    }
    // keep this CTA's shared memory alive until every peer has read it
    cluster.sync();
}

// One thread per sequence: pick the winning path and the next token.
__global__ void accept_select_kernel(const AcceptParams p) {
    griddep_wait();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= p.B) return;
    const int n_q = p.n_q;
    const int32_t* acc = p.ws_accept + (int64_t)b * n_q;
    int n_children[kAcceptMaxNq];
    for (int i = 0; i < n_q; ++i) n_children[i] = 0;
    for (int i = 1; i < n_q; ++i) n_children[parent_of(p, b, i)]++;
    int best_len = -1, best_leaf = 0;
    for (int leaf = 0; leaf < n_q; ++leaf) {
        if (n_children[leaf] != 0) continue;
        int nodes[kAcceptMaxNq];
        int depth = 0;
        for (int v = leaf; v != 0; v = parent_of(p, b, v)) nodes[depth++] = v;
        int len = 0;
        while (len < depth && acc[nodes[depth - 1 - len]]) ++len;
        if (len > best_len) { best_len = len; best_leaf = leaf; }
    }
    int nodes[kAcceptMaxNq];
    int depth = 0;
    for (int v = best_leaf; v != 0; v = parent_of(p, b, v)) nodes[depth++] = v;
    const int e = best_len > 0 ? nodes[depth - best_len] : 0;
    p.n_accepted[b] = best_len;
    p.next_token[b] = p.ws_sample[(int64_t)b * n_q + e];
    if (p.path) {
        for (int k = 0; k < n_q; ++k)
            p.path[(int64_t)b * n_q + k] = k < best_len ? nodes[depth - 1 - k] : -1;
    }
    if (p.diag) {
        for (int c = 0; c < 5; ++c) p.diag[(int64_t)b * n_q * 5 + c] = 0.f;
    }
}

template <int F>
cudaError_t launch_rows(const AcceptParams& p, int C, cudaStream_t st) {
    auto kern = accept_rows_kernel<F>;
    const size_t smem = (size_t)p.chunk * 8;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (C > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C, p.B * p.n_q, 1);
    cfg.blockDim = dim3(kNT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int F>
cudaError_t max_clusters(int C, int chunk, int* out) {
    auto kern = accept_rows_kernel<F>;
    const size_t smem = (size_t)chunk * 8;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (C > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C, 1, 1);
    cfg.blockDim = dim3(kNT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(out, kern, &cfg);
}

#define RAPID_ACCEPT_DISPATCH(FN, F_, ...)             \
    switch (F_) {                                      \
        case 1: return FN<1>(__VA_ARGS__);             \
        case 2: return FN<2>(__VA_ARGS__);             \
        case 3: return FN<3>(__VA_ARGS__);             \
        case 4: return FN<4>(__VA_ARGS__);             \
        case 5: return FN<5>(__VA_ARGS__);             \
        case 6: return FN<6>(__VA_ARGS__);             \
        case 7: return FN<7>(__VA_ARGS__);             \
        case 8: return FN<8>(__VA_ARGS__);             \
        case 9: return FN<9>(__VA_ARGS__);             \
        case 10: return FN<10>(__VA_ARGS__);           \
        case 11: return FN<11>(__VA_ARGS__);           \
        case 12: return FN<12>(__VA_ARGS__);           \
        case 13: return FN<13>(__VA_ARGS__);           \
        case 14: return FN<14>(__VA_ARGS__);           \
        case 15: return FN<15>(__VA_ARGS__);           \
        case 16: return FN<16>(__VA_ARGS__);           \
        default: return cudaErrorNotSupported;         \
    }

cudaError_t max_clusters_dispatch(int F, int C, int chunk, int* out) {
    RAPID_ACCEPT_DISPATCH(max_clusters, F, C, chunk, out)
}

cudaError_t launch_rows_dispatch(int F, const AcceptParams& p, int C, cudaStream_t st) {
    RAPID_ACCEPT_DISPATCH(launch_rows, F, p, C, st)
}

}  // namespace

AcceptShape accept_shape(int V, int preferred_cluster) {
    AcceptShape sh{};
    sh.vocab = V;
    int C = (V + kNT * 32 - 1) / (kNT * 32);
    if (preferred_cluster > 0) C = preferred_cluster;
    if (C < 1) C = 1;
    if (C > 16) C = 16;
    for (;;) {
        const int chunk = ((V + C - 1) / C + 3) / 4 * 4;
        const int F = (chunk + 4 * kNT - 1) / (4 * kNT);
        sh.cluster = C;
        sh.chunk = chunk;
        sh.F = F;
        if (F <= 16 || C >= 16) break;
        ++C;
    }
    return sh;
}

cudaError_t accept_check_cluster(AcceptShape* sh) {
    // Shrink the cluster until the hardware can co-schedule one of it.
    for (;;) {
        int n = 0;
        cudaError_t e = max_clusters_dispatch(sh->F, sh->cluster, sh->chunk, &n);
        if (e == cudaSuccess && n > 0) return cudaSuccess;
        (void)cudaGetLastError();
        if (sh->cluster <= 1) return e == cudaSuccess ? cudaErrorNotSupported : e;
        // next smaller power-of-two-ish size with the same row coverage
        const int C = sh->cluster > 8 ? 8 : sh->cluster / 2;
        sh->cluster = C;
        sh->chunk = ((sh->vocab + C - 1) / C + 3) / 4 * 4;
        sh->F = (sh->chunk + 4 * kNT - 1) / (4 * kNT);
        if (sh->F > 16) return cudaErrorNotSupported;
    }
}

cudaError_t launch_accept(const AcceptParams& p, const AcceptShape& sh, cudaStream_t st) {
    cudaError_t e = launch_rows_dispatch(sh.F, p, sh.cluster, st);
    if (e != cudaSuccess) return e;
    const int threads = 64;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((p.B + threads - 1) / threads, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, accept_select_kernel, p);
}

}  // namespace rapid
