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
// Layout of the work.  A row of V entries is cut into C slices, one per CTA
// of a thread-block cluster; the clusters are persistent and cluster c takes
// rows c, c + nclusters, ...  Each CTA keeps its slice of a row's (z, q) in
// shared memory, filled by bulk (TMA) copies.  A row needs two
// vocabulary-wide reductions -- the softmax of z/T and the softmax of the
// augmented logits -- which every CTA completes from the C slice partials
// that its peers send it with st.async into its shared memory (completion on
// an mbarrier).  Each CTA runs two warp groups on alternate rows, half a row
// apart, so that one computes while the other waits on the cluster; a row's
// buffer is refilled as soon as its second pass is done.  The rows kernel
// leaves the ratio-test outcomes and each row's softmax statistics; the
// selection kernel (one cluster per sequence) walks the chain or tree, picks
// n_accepted, and draws the next token from the one row it needs.
//
// Exponentials are taken against one reference per warp: the warp's max of x
// for p, and for the augmented logits a = x + eta (q - p) the bound
// max x + eta (a <= x + eta since q <= 1 and p >= 0; for eta > 32, where
// exp(a - bound) could underflow, the warp's exact max of a).  Sums carry
// their reference and are rescaled when combined.
#include <cooperative_groups.h>

#include <mutex>

#include "accept.cuh"
#include "common.cuh"

namespace cg = cooperative_groups;

namespace rapid {

namespace {

constexpr int kRT = kAcceptRowThreads;
constexpr int kST = kAcceptSelThreads;
constexpr int kSW = kST / 32;
// float4 groups per lane run in the draw: a warp segment of a slice of at
// most kAcceptMaxSlice entries is at most this many 128-entry blocks
constexpr int kRunF4 = (kAcceptMaxSlice + kSW * 128 - 1) / (kSW * 128);
constexpr size_t kSmemBudget = (size_t)2 * kAcceptMaxSlice * 8;   // dynamic shared memory for the row ring
constexpr int kMinSlice = 1024;          // rows shorter than C x this use fewer slices
constexpr int kSelSlice = 2048;          // selection: entries per CTA, at least
constexpr int kSelPerSm = 3;             // selection CTAs resident per SM (its launch bounds)
constexpr float kEtaBound = 32.f;        // largest eta for which max x + eta is the reference of a

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two-lane packed fp32 arithmetic (one instruction for both lanes).
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// Max over the 32 lanes (all lanes active), the same in every lane.
__device__ __forceinline__ float redux_max(float v) {
    float d;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(d) : "f"(v));
    return d;
}

struct MS {
    float m, s;   // a sum of exp(x - m)
};

// Combine the (m, s) of the 32 lanes; the result is the same in every lane.
__device__ __forceinline__ MS warp_ms(MS v) {
    const float m = redux_max(v.m);
    const float s = v.s > 0.f ? v.s * ex2((v.m - m) * kLog2e) : 0.f;
    return MS{m, warp_sum(s)};
}

constexpr int kGroups = 2;               // warp groups of a row-kernel CTA, one row each
constexpr int kGT = kRT / kGroups;       // threads of a group
constexpr int kGW = kGT / 32;            // warps of a group

struct RowsShared {
    uint64_t zfull[kGroups];  // the z half of the group's slice landed (pass 1 needs only z)
    uint64_t full[kGroups];   // the q half landed
    uint64_t mb1[kGroups];    // slice partials of reduction 1 received
    uint64_t mb2[kGroups];    // slice partials of reduction 2 received
    uint64_t stagger;         // group 0 is past its first reduction 1: group 1 may start
    float2 recv1[kGroups][kAcceptMaxCluster];   // (m, s) of x per slice
    float2 recv2[kGroups][kAcceptMaxCluster];   // (reference, s) of a per slice
    float recv2a[kGroups][kAcceptMaxCluster];   // max of a per slice
    float2 red1[kGroups][kGW];   // per-warp partials of the group's row
    float2 red2[kGroups][kGW];
    float red2a[kGroups][kGW];
    int arrived[kGroups][2];     // warps of the group done with pass 1, pass 2
    int abort;                   // a wait gave up: stop waiting, let the kernel run out
};

// The Philox key of the call: the host's value, or the one in device memory
// now (read through L2: an earlier kernel of the stream may have changed it;
// both kernels read it only after griddep_wait()).
__device__ __forceinline__ uint2 philox_key(const AcceptParams& p) {
    if (!p.seed_dev) return make_uint2(p.seed_lo, p.seed_hi);
    const unsigned long long s = __ldcg(p.seed_dev);
    return make_uint2((uint32_t)(s & 0xffffffffull), (uint32_t)(s >> 32));
}

// Nodes of sequence b: n_q, or the caller's count clamped to [1, n_q].  The
// nodes past it are padding: no one's children, never on a path.
__device__ __forceinline__ int node_count(const AcceptParams& p, int b) {
    if (!p.n_nodes) return p.n_q;
    const int n = p.n_nodes[b];
    return n < 1 ? 1 : (n > p.n_q ? p.n_q : n);
}

__device__ __forceinline__ int parent_of(const AcceptParams& p, int b, int i) {
    if (!p.parent) return i - 1;
    int par = p.parent[(int64_t)b * p.n_q + i];
    if (par < 0) par = 0;
    if (par > i - 1) par = i - 1;
    return par;
}

__device__ __forceinline__ void group_sync(int g) {
    asm volatile("bar.sync %0, %1;" ::"r"(1 + g), "r"(kGT) : "memory");
}

// A warp of the group is done with a phase (its slot written by lane 0):
// true, in every lane, for the last warp of the group to get there, which
// then sees every warp's slot.  The counter is reset by that warp.
__device__ __forceinline__ bool group_arrive(int* counter) {
    const int lane = threadIdx.x & 31;
    int last = 0;
    if (lane == 0) {
        __threadfence_block();
        last = atomicAdd(counter, 1) == kGW - 1;
        if (last) {
            *counter = 0;
            __threadfence_block();
        }
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    __syncwarp();
    return last != 0;
}

// Split cluster barrier: arrive (no ordering) and wait, by every thread.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t mapa_u32(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_async_v2(uint32_t raddr, float a, float b, uint32_t rbar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(raddr),
        "f"(a), "f"(b), "r"(rbar)
        : "memory");
}
__device__ __forceinline__ void st_async_f32(uint32_t raddr, float a, uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(raddr),
                 "f"(a), "r"(rbar)
                 : "memory");
}

// Bounded wait on an mbarrier phase.  After a wait gave up (one second), the
// CTA stops waiting altogether; the error word records where.
__device__ __forceinline__ void wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort,
                                              unsigned int* err, unsigned int code) {
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = global_timer_ns();
    while (!*abort) {
        if (mbar_try_wait_sleep(bar, parity, 1000u)) return;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            if (err) {
                atomicOr(err, kErrWaitTimeout);
                atomicCAS(err + 1, 0u, code | 0x80000000u);
            }
            return;
        }
    }
}

// Per-thread state of the row a group works on.
template <int F>
struct RowState {
    float e[4 * F];   // exp(x - mw) of this thread's entries (x = z / T)
    float mw;         // warp max of x
    float fw;         // exp(mw - m1) / s1: p = e * fw
    float m1, s1;     // row softmax statistics of x (after reduction 1)
};

// Group thread t owns float4 groups t, t + kGT, ... of a row array of G groups (G
// a multiple of 32, so validity is warp-uniform).  Entries past the slice
// hold z = -inf and q = 0, which give p = 0, h = 0 and a residual weight of
// 0, so the passes need no per-entry bounds checks.
template <int F>
__device__ __forceinline__ bool group_valid(int f, int G) {
    return f < F - 1 || (int)(threadIdx.x % kGT) + f * kGT < G;
}

// Pass 1: x = z / T; exp(x - mw) with mw the warp max; the warp's (mw, sum).
template <int F>
__device__ __forceinline__ MS pass1(RowState<F>& st, const float* zb, int G, float invT) {
    const int t = threadIdx.x % kGT;
    const float2 it2 = make_float2(invT, invT);
    float mt = -INFINITY;
#pragma unroll
    for (int f = 0; f < F; ++f) {
        if (group_valid<F>(f, G)) {
            const float4 r = *reinterpret_cast<const float4*>(zb + 4 * (t + f * kGT));
            const float2 x01 = mul2(make_float2(r.x, r.y), it2);
            const float2 x23 = mul2(make_float2(r.z, r.w), it2);
            st.e[4 * f] = x01.x; st.e[4 * f + 1] = x01.y;
            st.e[4 * f + 2] = x23.x; st.e[4 * f + 3] = x23.y;
            mt = max3(mt, x01.x, x01.y);
            mt = max3(mt, x23.x, x23.y);
        }
    }
    const float mw = redux_max(mt);
    const float mb = mw == -INFINITY ? 0.f : mw * kLog2e;
    const float2 l2 = make_float2(kLog2e, kLog2e), nb = make_float2(-mb, -mb);
    float2 s = make_float2(0.f, 0.f);
#pragma unroll
    for (int f = 0; f < F; ++f) {
        if (group_valid<F>(f, G)) {
            const float2 g01 = fma2(make_float2(st.e[4 * f], st.e[4 * f + 1]), l2, nb);
            const float2 g23 = fma2(make_float2(st.e[4 * f + 2], st.e[4 * f + 3]), l2, nb);
            const float2 e01 = make_float2(ex2(g01.x), ex2(g01.y));
            const float2 e23 = make_float2(ex2(g23.x), ex2(g23.y));
            st.e[4 * f] = e01.x; st.e[4 * f + 1] = e01.y;
            st.e[4 * f + 2] = e23.x; st.e[4 * f + 3] = e23.y;
            s = add2(s, e01);
            s = add2(s, e23);
        }
    }
    st.mw = mw;
    return MS{mw, warp_sum(s.x + s.y)};
}

// Pass 2: p = e * fw; a = x + eta (q - p); the warp's (rw, sum of exp(a - rw))
// and its max of a.
template <int F>
__device__ __forceinline__ MS pass2(RowState<F>& st, const float* zb, const float* qb, int G,
                                    float invT, float eta, float* amax_w) {
    const int t = threadIdx.x % kGT;
    const float fw = st.mw == -INFINITY ? 0.f : ex2((st.mw - st.m1) * kLog2e) / st.s1;
    st.fw = fw;
    const float2 it2 = make_float2(invT, invT), nf2 = make_float2(-fw, -fw);
    const float2 eta2 = make_float2(eta, eta);
    float rw;
    if (eta <= kEtaBound) {
        rw = st.mw == -INFINITY ? -INFINITY : st.mw + eta;
    } else {
        float am = -INFINITY;
#pragma unroll
        for (int f = 0; f < F; ++f) {
            if (group_valid<F>(f, G)) {
                const int el = 4 * (t + f * kGT);
                const float4 z4 = *reinterpret_cast<const float4*>(zb + el);
                const float4 q4 = *reinterpret_cast<const float4*>(qb + el);
                const float2 a01 = fma2(eta2, fma2(make_float2(st.e[4 * f], st.e[4 * f + 1]), nf2,
                                                   make_float2(q4.x, q4.y)),
                                        mul2(make_float2(z4.x, z4.y), it2));
                const float2 a23 = fma2(eta2, fma2(make_float2(st.e[4 * f + 2], st.e[4 * f + 3]), nf2,
                                                   make_float2(q4.z, q4.w)),
                                        mul2(make_float2(z4.z, z4.w), it2));
                am = max3(am, a01.x, a01.y);
                am = max3(am, a23.x, a23.y);
            }
        }
        rw = redux_max(am);
    }
    const float rb = rw == -INFINITY ? 0.f : rw * kLog2e;
    const float2 l2 = make_float2(kLog2e, kLog2e), nb = make_float2(-rb, -rb);
    float amax = -INFINITY;
    float2 s = make_float2(0.f, 0.f);
#pragma unroll
    for (int f = 0; f < F; ++f) {
        if (group_valid<F>(f, G)) {
            const int el = 4 * (t + f * kGT);
            const float4 z4 = *reinterpret_cast<const float4*>(zb + el);
            const float4 q4 = *reinterpret_cast<const float4*>(qb + el);
            const float2 a01 = fma2(eta2, fma2(make_float2(st.e[4 * f], st.e[4 * f + 1]), nf2,
                                               make_float2(q4.x, q4.y)),
                                    mul2(make_float2(z4.x, z4.y), it2));
            const float2 a23 = fma2(eta2, fma2(make_float2(st.e[4 * f + 2], st.e[4 * f + 3]), nf2,
                                               make_float2(q4.z, q4.w)),
                                    mul2(make_float2(z4.z, z4.w), it2));
            amax = max3(amax, a01.x, a01.y);
            amax = max3(amax, a23.x, a23.y);
            const float2 g01 = fma2(a01, l2, nb);
            const float2 g23 = fma2(a23, l2, nb);
            // same pairing and order of additions as pass 1, so that eta = 0
            // gives p_hat == p bit for bit
            s = add2(s, make_float2(ex2(g01.x), ex2(g01.y)));
            s = add2(s, make_float2(ex2(g23.x), ex2(g23.y)));
        }
    }
    *amax_w = redux_max(amax);
    return MS{rw, warp_sum(s.x + s.y)};
}

template <int F>
__global__ void __launch_bounds__(kRT, 1)
accept_rows_kernel(const AcceptParams p) {
    cg::cluster_group cluster = cg::this_cluster();
    const int C = p.C;
    const int G = p.groups;
    const int span = 4 * G;
    const int rank = (int)cluster.block_rank();
    const int cid = (int)(blockIdx.x / C);
    const int t = threadIdx.x;
    const int g = t / kGT;           // warp group: local rows g, g + 2, g + 4, ...
    const int tg = t % kGT;
    const int wg = tg >> 5, lane = t & 31;

    extern __shared__ float4 dyn_f4[];
    float* bufs = reinterpret_cast<float*>(dyn_f4);
    __shared__ RowsShared sh;

    const int64_t lo = (int64_t)rank * p.chunk;
    int64_t n64 = (int64_t)p.V - lo;
    if (n64 > p.chunk) n64 = p.chunk;
    if (n64 < 0) n64 = 0;
    const int n = (int)n64;
    const int nrows = cid < p.rows ? (p.rows - cid + p.nclusters - 1) / p.nclusters : 0;

    if (t == 0) {
        for (int i = 0; i < kGroups; ++i) {
            mbar_init(&sh.zfull[i], 1);
            mbar_init(&sh.full[i], 1);
            mbar_init(&sh.mb1[i], 1);
            mbar_init(&sh.mb2[i], 1);
            sh.arrived[i][0] = sh.arrived[i][1] = 0;
        }
        mbar_init(&sh.stagger, 1);
        sh.abort = 0;
        fence_mbar_init();
    }
    // padding past the slice: z = -inf, q = 0 (bulk copies never write there)
    for (int b = 0; b < kGroups; ++b) {
        float* zb = bufs + (size_t)b * 2 * span;
        for (int e = n + t; e < span; e += kRT) {
            zb[e] = -INFINITY;
            zb[span + e] = 0.f;
        }
    }
    cluster.sync();   // barriers and padding in place before any copy or peer send
    griddep_wait();

    float* zb = bufs + (size_t)g * 2 * span;   // this group's row buffer
    float* qb = zb + span;
    auto row_of = [&](int i) -> int64_t { return cid + (int64_t)i * p.nclusters; };
    // A row of a node past its sequence's node count is padding: every CTA of
    // the cluster skips it alike (no copy, no exchange, no result).
    auto padding = [&](int i) -> bool {
        if (!p.n_nodes) return false;
        const int64_t row = row_of(i);
        const int b = (int)(row / p.n_q);
        return (int)(row - (int64_t)b * p.n_q) >= node_count(p, b);
    };
    // The group's first row at or after i that is not padding (i, i + 2, ...),
    // or nrows.  Padding rows take no buffer phase: the k-th real row of the
    // group is the k-th phase of its buffer barrier, so a warp can never wait
    // on a phase two ahead of the barrier (which would pass at once, on the
    // phase before).
    auto next_real = [&](int i) -> int {
        while (i < nrows && padding(i)) i += 2;
        return i;
    };
    auto load_row = [&](int i) {      // one thread, bulk path, a row that is not padding
        mbar_arrive_expect_tx(&sh.zfull[g], (uint32_t)(n * 4));
        mbar_arrive_expect_tx(&sh.full[g], (uint32_t)(n * 4));
        if (n > 0) {
            // rows are read once here (the selection re-reads at most one row
            // of a sequence, which it prefetches itself): evict-first, so the
            // stream does not push the selection's code and inputs out of L2
            const int64_t off = row_of(i) * p.V + lo;
            const uint64_t pol = l2_policy_evict_first();
            bulk_g2s_hint(zb, p.z + off, (uint32_t)(n * 4), &sh.zfull[g], pol);
            bulk_g2s_hint(qb, p.q + off, (uint32_t)(n * 4), &sh.full[g], pol);
        }
    };
    // L2 prefetch of a later row of this group, so that its bulk copy, issued
    // only once the buffer is free, is served from L2
    auto prefetch_row = [&](int i) {   // one thread, bulk path, a real row or nrows
        if (i < nrows && n > 0) {
            const int64_t off = row_of(i) * p.V + lo;
            bulk_prefetch_l2(p.z + off, (uint32_t)(n * 4));
            bulk_prefetch_l2(p.q + off, (uint32_t)(n * 4));
        }
    };
    if (p.bulk && tg == 0) {
        const int j0 = next_real(g);
        if (j0 < nrows) load_row(j0);
    }

    // The group's last two warps run the ratio tests: thread tg handles child
    // c = tg - (kGT - kAcceptMaxNq).  Its token and parent are loaded a row ahead.
    const int c = tg - (kGT - kAcceptMaxNq);
    const bool rt_thread = c >= 0 && c < p.n_q;
    int pf_tok = -1, pf_par = -1;
    auto prefetch_node = [&](int i) {
        if (rt_thread && i < nrows) {
            const int b = (int)(row_of(i) / p.n_q);
            pf_tok = p.tokens[(int64_t)b * p.n_q + c];
            pf_par = c == 0 ? -1 : parent_of(p, b, c);
        }
    };
    prefetch_node(g);

    RowState<F> st;
    // Each row: its copy lands, pass 1, reduction 1 across the cluster, pass 2,
    // reduction 2, then the ratio tests and the residual mass.  Warps move on
    // independently; the last warp of a phase combines the group's partials
    // and sends them to the cluster, and every warp waits for the cluster's
    // partials itself.  The other group computes while this one waits.
    // kx counts the group's rows that are not padding: the phase of zfull[g],
    // full[g], mb1[g] and mb2[g] for the row at hand.
    int kx = 0;
#pragma unroll 1
    for (int i = g; i < nrows; i += 2) {
        const int64_t row = row_of(i);
        const int b = (int)(row / p.n_q);
        const int j = (int)(row - (int64_t)b * p.n_q);
        if (padding(i)) {   // no copy, no exchange, no buffer phase
            prefetch_node(i + 2);
            if (tg == 0 && i == 0) mbar_arrive(&sh.stagger);
            continue;
        }
        if (tg == 0) {
            // arm this row's exchange barriers (their previous phases completed
            // before any warp of the group could finish the previous row)
            mbar_arrive_expect_tx(&sh.mb1[g], (uint32_t)(C * 8));
            mbar_arrive_expect_tx(&sh.mb2[g], (uint32_t)(C * 12));
            if (p.bulk) prefetch_row(next_real(i + 2));
        }
        const int my_tok = pf_tok, my_par = pf_par;
        prefetch_node(i + 2);
        // the groups run half a row apart, so that one computes while the
        // other waits on the cluster
        if (i == 1)
            wait_or_abort(&sh.stagger, 0u, &sh.abort, p.err, 0x06000000u);
        if (p.bulk) {
            // pass 1 reads only z; q keeps landing meanwhile
            wait_or_abort(&sh.zfull[g], (uint32_t)(kx & 1), &sh.abort, p.err,
                          0x01000000u | (unsigned)(i & 0xffff));
        } else {
            const int64_t off = row * p.V + lo;
            for (int e = tg; e < n; e += kGT) {
                zb[e] = p.z[off + e];
                qb[e] = p.q[off + e];
            }
            group_sync(g);
        }
        // z and q at the token of child c of this row, for its ratio test (q
        // once its half has landed, before pass 2)
        int key = -1;
        float2 zq = make_float2(0.f, 0.f);
        if (rt_thread && c > j && my_par == j) {
            if (my_tok < 0 || my_tok >= p.V) {
                key = rank == 0 ? -2 : -1;
            } else if (my_tok >= lo && my_tok < lo + n) {
                key = my_tok;
                zq.x = zb[my_tok - lo];
            }
        }
        // pass 1; the group's last warp sends the slice's (m, s) to the cluster
        {
            const MS w1 = pass1<F>(st, zb, G, p.invT);
            if (lane == 0) sh.red1[g][wg] = make_float2(w1.m, w1.s);
            if (group_arrive(&sh.arrived[g][0])) {
                const float2 x = lane < kGW ? sh.red1[g][lane] : make_float2(-INFINITY, 0.f);
                const MS c1 = warp_ms(MS{x.x, x.y});
                if (lane < C)
                    st_async_v2(mapa_u32(smem_u32(&sh.recv1[g][rank]), (uint32_t)lane), c1.m, c1.s,
                                mapa_u32(smem_u32(&sh.mb1[g]), (uint32_t)lane));
            }
        }
        // uniform r_c of the ratio test, while the cluster reduces
        float r_c = 0.f;
        if (key >= 0) {
            const uint2 key = philox_key(p);
            const Philox4 rnd = philox4x32_10((uint32_t)c, (uint32_t)b, 0u, 0u, key.x, key.y);
            r_c = word_uniform(rnd.w[0]);
        }
        wait_or_abort(&sh.mb1[g], (uint32_t)(kx & 1), &sh.abort, p.err,
                      0x03000000u | (unsigned)(i & 0xffff));
        {
            MS r1{-INFINITY, 0.f};
            if (lane < C) r1 = MS{sh.recv1[g][lane].x, sh.recv1[g][lane].y};
            r1 = warp_ms(r1);
            st.m1 = r1.m;
            st.s1 = r1.s;
        }
        if (i == 0 && tg == 0) mbar_arrive(&sh.stagger);
        if (p.bulk)
            wait_or_abort(&sh.full[g], (uint32_t)(kx & 1), &sh.abort, p.err,
                          0x04000000u | (unsigned)(i & 0xffff));
        if (key >= 0) zq.y = qb[key - lo];
        // pass 2; the group's last warp sends the slice's (reference, s, max a)
        {
            float amw;
            const MS w2 = pass2<F>(st, zb, qb, G, p.invT, p.eta, &amw);
            if (lane == 0) {
                sh.red2[g][wg] = make_float2(w2.m, w2.s);
                sh.red2a[g][wg] = amw;
            }
            if (group_arrive(&sh.arrived[g][1])) {
                const float2 x = lane < kGW ? sh.red2[g][lane] : make_float2(-INFINITY, 0.f);
                const MS c2 = warp_ms(MS{x.x, x.y});
                const float ac = redux_max(lane < kGW ? sh.red2a[g][lane] : -INFINITY);
                if (lane < C) {
                    const uint32_t rbar = mapa_u32(smem_u32(&sh.mb2[g]), (uint32_t)lane);
                    st_async_v2(mapa_u32(smem_u32(&sh.recv2[g][rank]), (uint32_t)lane), c2.m, c2.s, rbar);
                    st_async_f32(mapa_u32(smem_u32(&sh.recv2a[g][rank]), (uint32_t)lane), ac, rbar);
                }
                if (lane == 0 && p.bulk) {
                    // every warp of the group is done with the buffer: it takes
                    // the group's next row while reduction 2 travels
                    const int jn = next_real(i + 2);
                    if (jn < nrows) {
                        fence_proxy_async_smem();
                        load_row(jn);
                    }
                }
            }
        }
        wait_or_abort(&sh.mb2[g], (uint32_t)(kx & 1), &sh.abort, p.err,
                      0x02000000u | (unsigned)(i & 0xffff));
        ++kx;
        float m2, s2;
        {
            MS r2{-INFINITY, 0.f};
            float am = -INFINITY;
            if (lane < C) {
                r2 = MS{sh.recv2[g][lane].x, sh.recv2[g][lane].y};
                am = sh.recv2a[g][lane];
            }
            r2 = warp_ms(r2);
            am = redux_max(am);
            // (m2, s2) with m2 the row max of a, so that max p_hat = 1 / s2
            m2 = am;
            s2 = r2.m == am ? r2.s : r2.s * ex2((r2.m - am) * kLog2e);
        }
        const float thr = p.clamp ? 0.1f / s2 : -1.0f;
        // ratio test of child c
        const int64_t node = (int64_t)b * p.n_q + c;
        if (key >= 0) {
            const float x = zq.x * p.invT;
            const float pt = ex2((x - st.m1) * kLog2e) / st.s1;
            const float a = fmaf(p.eta, zq.y - pt, x);
            float ph = ex2((a - m2) * kLog2e) / s2;
            if (ph < thr) ph = pt;
            const float ratio = zq.y == 0.f ? INFINITY : ph / zq.y;
            p.ws_accept[node] = r_c <= fminf(1.0f, ratio) ? 1 : 0;
            if (p.diag) {
                float* dg = p.diag + node * 5;
                dg[0] = pt; dg[1] = ph; dg[2] = zq.y; dg[3] = ratio; dg[4] = r_c;
            }
        } else if (key == -2) {
            p.ws_accept[node] = 0;   // token outside the vocabulary: reject
        }
        if (rank == 0 && tg == 0) {
            float* sts = p.ws_stats + row * 4;
            sts[0] = st.m1; sts[1] = st.s1; sts[2] = m2; sts[3] = s2;
        }
        if (!p.bulk) group_sync(g);   // the synchronous copy of the next row overwrites the buffer
    }
    __syncthreads();   // both groups done: no copy of this CTA is outstanding unless a wait gave up
    if (t == 0) {
        griddep_launch_dependents();
        if (p.bulk && sh.abort) {
            // a wait gave up: let the groups' last copies land before the CTA exits
            for (int gg = 0; gg < kGroups; ++gg) {
                int nmine = 0;   // the group's real rows: one buffer phase each
                for (int i = gg; i < nrows; i += 2) nmine += padding(i) ? 0 : 1;
                if (nmine > 0) {
                    mbar_wait(&sh.zfull[gg], (uint32_t)((nmine - 1) & 1), nullptr);
                    mbar_wait(&sh.full[gg], (uint32_t)((nmine - 1) & 1), nullptr);
                }
            }
        }
    }
    // no CTA leaves while a peer may still deliver into its shared memory
    cluster.sync();
}

// Selection, one thread-block cluster per sequence b, one CTA per vocabulary
// slice.  Every CTA picks the winning path (from a few hundred bytes) and
// the last accepted node e, then weights its slice of row e for the draw of
// the next token by inverse CDF in token-id order with u_{e+1}: the residual
// max(p - p_hat, p - q, 0) if e has children (a rejection happened below it),
// else p (the bonus draw; also the fallback when the residual has no mass).
// The weights stay in the CTA's shared memory; each CTA stores its slice
// total into every peer's table (distributed shared memory, one cluster
// barrier), and in the CTA whose slice holds the target one warp finds the
// warp segment that holds it, then the entry, 128 entries at a time.
__device__ __forceinline__ float resid_weight(float z, float qk, float invT, float eta, float m1,
                                              float inv_s1, float m2, float inv_s2, float thr) {
    const float x = z * invT;
    const float pk = ex2((x - m1) * kLog2e) * inv_s1;
    const float a = fmaf(eta, qk - pk, x);
    float ph = ex2((a - m2) * kLog2e) * inv_s2;
    if (ph < thr) ph = pk;
    return pk - min3(pk, ph, qk);   // max(p - p_hat, p - q, 0)
}

// Float4 group i of the weights (entries i .. i + 3, i a multiple of 4);
// entries at or past a1 read as 0.
__device__ __forceinline__ float4 run_f4(const float* sw, int i, int a1) {
    float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i + 3 < a1) {
        w = *reinterpret_cast<const float4*>(sw + i);
    } else if (i < a1) {
        w.x = sw[i];
        if (i + 1 < a1) w.y = sw[i + 1];
        if (i + 2 < a1) w.z = sw[i + 2];
    }
    return w;
}

__global__ void __launch_bounds__(kST, 3) accept_select_kernel(const AcceptParams p) {
    cg::cluster_group cluster = cg::this_cluster();
    extern __shared__ float4 sel_dyn[];
    float* sw = reinterpret_cast<float*>(sel_dyn);   // [chunk] weights of this slice
    __shared__ int s_acc[kAcceptMaxNq], s_par[kAcceptMaxNq], s_kids[kAcceptMaxNq];
    __shared__ int s_key[2];
    __shared__ int s_e, s_has_children, s_depth, s_len;
    __shared__ int s_nodes[kAcceptMaxNq];   // the winning path, leaf first
    __shared__ float s_seg[kSW];   // weight total of each warp's segment
    __shared__ float s_run[kSW][32], s_runi[kSW][32];   // lane runs of each segment: sums, inclusive prefix
    __shared__ float s_tot[2][kAcceptMaxCluster];   // every slice's total, per round
    __shared__ float4 s_stats[kAcceptMaxNq];   // every row's (m1, s1, m2, s2), read up front

    const int cs = (int)cluster.block_rank();   // vocabulary slice
    const int b = blockIdx.y;
    const int t = threadIdx.x;
    const int warp = t >> 5, lane = t & 31;
    const int n_q = p.n_q;
    cluster_arrive();   // this CTA has started; peers wait for it before storing into it
    griddep_wait();
    // the next kernel of the stream may launch now: whatever it does before
    // its own griddep_wait() touches no memory this grid reads or writes
    griddep_launch_dependents();
    const int nn = node_count(p, b);   // nodes of this sequence
    // Device-side inputs the host cannot check (clamped or rejected on the
    // way, so memory stays safe): a node count outside [1, n_q], a parent
    // outside [0, i) or a draft token outside the vocabulary sets the
    // bad-input bit of the error word (one CTA of the cluster looks).
    if (cs == 0 && t < n_q && p.err) {
        bool bad = false;
        if (t == 0) {
            if (p.n_nodes) {
                const int c = p.n_nodes[b];
                bad = c < 1 || c > n_q;
            }
        } else if (t < nn) {
            const int tok = p.tokens[(int64_t)b * n_q + t];
            bad = tok < 0 || tok >= p.V;
            if (p.parent) {
                const int par = p.parent[(int64_t)b * n_q + t];
                bad = bad || par < 0 || par >= t;
            }
        }
        if (bad) atomicOr(p.err, kErrBadInput);
    }
    if (t < n_q) {
        s_acc[t] = t == 0 ? 1 : p.ws_accept[(int64_t)b * n_q + t];
        s_par[t] = t == 0 ? -1 : parent_of(p, b, t);
        s_kids[t] = 0;
        s_stats[t] = reinterpret_cast<const float4*>(p.ws_stats)[(int64_t)b * n_q + t];
    }
    __syncthreads();
    if (t > 0 && t < nn) s_kids[s_par[t]] = 1;   // every writer stores the same value
    __syncthreads();

    // every leaf: the number of accepted nodes from the root down its path
    int key = -1;
    if (t < nn) {
        if (!s_kids[t]) {   // a leaf
            // one walk up: the depth, and the steps from the leaf to the
            // rejected node nearest the root (the path's first rejection)
            int steps = 0, rej = -1;
            for (int v = t; v != 0; v = s_par[v], ++steps)
                if (!s_acc[v]) rej = steps;
            const int len = rej < 0 ? steps : steps - rej - 1;
            key = (len << 8) | (255 - t);   // most accepted, then smallest leaf
        }
    }
    if (warp < 2) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, o));
        if (lane == 0) s_key[warp] = key;
    }
    __syncthreads();
    if (t == 0) {
        const int best = max(s_key[0], s_key[1]);
        const int best_len = best >> 8, best_leaf = 255 - (best & 255);
        int depth = 0;
        for (int v = best_leaf; v != 0; v = s_par[v]) s_nodes[depth++] = v;   // the leaf first
        const int e = best_len > 0 ? s_nodes[depth - best_len] : 0;
        s_depth = depth;
        s_len = best_len;
        s_e = e;
        s_has_children = s_kids[e];
    }
    __syncthreads();
    // the outputs (cluster rank 0), one path entry per thread
    if (cs == 0 && t < n_q) {
        const int len = s_len;
        if (t == 0) p.n_accepted[b] = len;
        if (p.path) p.path[(int64_t)b * n_q + t] = t < len ? s_nodes[s_depth - 1 - t] : -1;
        if (p.diag && t < 5) p.diag[(int64_t)b * n_q * 5 + t] = 0.f;   // the root's row
    }

    const int e = s_e;
    // the uniform of the draw, u_{e+1}: warp 0 needs it after the exchange
    float u = 0.f;
    if (warp == 0) {
        const uint2 key = philox_key(p);
        const Philox4 rnd = philox4x32_10((uint32_t)(e + 1), (uint32_t)b, 0u, 0u, key.x, key.y);
        u = word_uniform(rnd.w[1]);
    }
    const int64_t row = (int64_t)b * n_q + e;
    const float4 sts = s_stats[e];
    const float m1 = sts.x, inv_s1 = 1.f / sts.y, m2 = sts.z, inv_s2 = 1.f / sts.w;
    const float thr = p.clamp ? 0.1f * inv_s2 : -1.0f;   // max p_hat = 1 / s2
    const int64_t lo = (int64_t)cs * p.chunk;
    int64_t n64 = (int64_t)p.V - lo;
    if (n64 > p.chunk) n64 = p.chunk;
    const int n = n64 > 0 ? (int)n64 : 0;
    const float* zr = p.z + row * p.V + lo;
    const float* qr = p.q + row * p.V + lo;
    // the slice of row e starts its trip to L2 in two bulk requests, so the
    // loads below wait for L2 rather than for DRAM one round trip at a time
    if (t == 0 && p.bulk && n > 0) {
        bulk_prefetch_l2(zr, (uint32_t)n * 4u);
        if (s_has_children) bulk_prefetch_l2(qr, (uint32_t)n * 4u);
    }

    // The residual if e has children, else p; p also when the residual has no
    // mass in any slice.  Warp w weights one contiguous segment [g0, g1) of
    // the slice (a multiple of 128 entries long, so float4 groups never
    // straddle two segments); its sum is the segment's total, which the
    // draw below uses without reading the weights again.
    bool resid = s_has_children != 0;
    const int seg = (n + kSW * 128 - 1) / (kSW * 128) * 128;
    const int g0 = min(n, warp * seg);
    const int g1 = min(n, g0 + seg);
    const int nf = seg / 128;   // float4 groups per lane run: at most kRunF4 (slices of at most kAcceptMaxSlice)
    int owner = -1;
    float tin = INFINITY;
    float segv = 0.f, segi = 0.f;   // warp 0: segment total and inclusive prefix, one per lane
    for (int round = 0;; ++round) {
        float acc = 0.f;
        if (p.bulk) {   // 16-byte aligned rows, n a multiple of 4
            const float4* z4 = reinterpret_cast<const float4*>(zr);
            const float4* q4 = reinterpret_cast<const float4*>(qr);
            float4* w4 = reinterpret_cast<float4*>(sw);
#pragma unroll 4
            for (int k = g0 / 4 + lane; k < g1 / 4; k += 32) {
                const float4 a = z4[k];
                float4 w;
                if (resid) {
                    const float4 c = q4[k];
                    w.x = resid_weight(a.x, c.x, p.invT, p.eta, m1, inv_s1, m2, inv_s2, thr);
                    w.y = resid_weight(a.y, c.y, p.invT, p.eta, m1, inv_s1, m2, inv_s2, thr);
                    w.z = resid_weight(a.z, c.z, p.invT, p.eta, m1, inv_s1, m2, inv_s2, thr);
                    w.w = resid_weight(a.w, c.w, p.invT, p.eta, m1, inv_s1, m2, inv_s2, thr);
                } else {
                    w.x = ex2((a.x * p.invT - m1) * kLog2e) * inv_s1;
                    w.y = ex2((a.y * p.invT - m1) * kLog2e) * inv_s1;
                    w.z = ex2((a.z * p.invT - m1) * kLog2e) * inv_s1;
                    w.w = ex2((a.w * p.invT - m1) * kLog2e) * inv_s1;
                }
                w4[k] = w;
                acc += (w.x + w.y) + (w.z + w.w);
            }
        } else {
#pragma unroll 4
            for (int k = g0 + lane; k < g1; k += 32) {
                const float w = resid ? resid_weight(zr[k], qr[k], p.invT, p.eta, m1, inv_s1, m2,
                                                     inv_s2, thr)
                                      : ex2((zr[k] * p.invT - m1) * kLog2e) * inv_s1;
                sw[k] = w;
                acc += w;
            }
        }
        acc = warp_sum(acc);
        if (lane == 0) s_seg[warp] = acc;
        // The draw's search tables, built while the cluster waits for its
        // slowest slice: each warp's segment in 32 contiguous lane runs of
        // nf float4 groups (sums and inclusive prefix), and in warp 0 the
        // segment totals with their inclusive prefix.
        __syncwarp();
        {
            const int r0 = g0 + lane * 4 * nf;
            float ls = 0.f;
#pragma unroll
            for (int j = 0; j < kRunF4; ++j) {
                if (j < nf) {
                    const float4 w = run_f4(sw, r0 + 4 * j, g1);
                    ls = (((ls + w.x) + w.y) + w.z) + w.w;
                }
            }
            float incl = ls;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            s_run[warp][lane] = ls;
            s_runi[warp][lane] = incl;
        }
        __syncthreads();
        // every CTA of the cluster has started (the arrival at entry) before
        // warp 0 stores this slice's total into each peer's table
        cluster_wait();
        if (warp == 0) {
            segv = lane < kSW ? s_seg[lane] : 0.f;
            const float tot = warp_sum(segv);
            if (lane < p.C) *cluster.map_shared_rank(&s_tot[round][cs], lane) = tot;
            segi = segv;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, segi, o);
                if (lane >= o) segi += y;
            }
        }
        cluster.sync();   // every table holds every slice's total; nothing remote is read after this
        // each warp reads the table: the totals, in slice order, are the same
        // bits in every warp and every CTA, and so is the decision to go on
        const float mc = lane < p.C ? s_tot[round][lane] : 0.f;
        const float totals = warp_sum(mc);
        if (resid && !(totals > 0.f)) {
            resid = false;
            cluster_arrive();   // pairs with the wait before the next round's stores
            continue;
        }
        if (warp != 0) return;
        const float target = u * totals;
        float incl = mc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, mc > 0.f && incl > target);
        const unsigned pos = __ballot_sync(0xffffffffu, mc > 0.f);
        if (hit) {
            owner = __ffs(hit) - 1;
            tin = target - __shfl_sync(0xffffffffu, incl - mc, owner);
        } else if (pos) {
            owner = 31 - __clz(pos);   // rounding left the target past the end
        }
        break;
    }
    // warp 0 alone from here
    if (owner < 0) {   // no mass at all (degenerate input)
        if (cs == 0 && lane == 0) p.next_token[b] = 0;
        return;
    }
    if (cs != owner) return;
    // the segment that holds the target, from the segment totals
    int ow = -1;
    float tw = INFINITY;
    {
        const unsigned hit = __ballot_sync(0xffffffffu, segv > 0.f && segi > tin);
        const unsigned pos = __ballot_sync(0xffffffffu, segv > 0.f);
        if (hit) {
            ow = __ffs(hit) - 1;
            tw = tin - __shfl_sync(0xffffffffu, segi - segv, ow);
        } else if (pos) {
            ow = 31 - __clz(pos);
        }
    }
    if (ow < 0) {   // the owner slice has no mass (rounding): its first entry
        if (lane == 0) p.next_token[b] = (int)lo;
        return;
    }
    // the run that holds the target (else, from rounding, the last run with
    // mass), then the first positive entry of that run whose running sum
    // passes the target, else the run's last positive entry
    const int a0 = ow * seg;
    const int a1 = min(n, a0 + seg);
    const int r0 = a0 + lane * 4 * nf;
    const float ls = s_run[ow][lane];
    const float incl = s_runi[ow][lane];
    const unsigned hit = __ballot_sync(0xffffffffu, ls > 0.f && incl > tw);
    const unsigned pos = __ballot_sync(0xffffffffu, ls > 0.f);
    const int src = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
    if (src < 0) {   // unreachable: the segment has mass
        if (lane == 0) p.next_token[b] = (int)(lo + a0);
        return;
    }
    const float tl = tw - __shfl_sync(0xffffffffu, incl - ls, src);
    if (lane != src) return;
    float ce = 0.f;
    int pick = -1, last = -1;
#pragma unroll
    for (int j = 0; j < kRunF4; ++j) {
        if (j < nf) {
            const int i = r0 + 4 * j;
            const float4 w = run_f4(sw, i, a1);
            const float c[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (c[k] > 0.f) {
                    last = i + k;
                    if (pick < 0 && ce + c[k] > tl) pick = i + k;
                }
                ce += c[k];
            }
        }
    }
    p.next_token[b] = (int)(lo + (pick >= 0 ? pick : last));
}

template <int F>
cudaError_t set_rows_attrs(int C, size_t smem) {
    auto kern = accept_rows_kernel<F>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (C > 8) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

size_t rows_smem(int groups, int nbuf) { return (size_t)nbuf * groups * 32; }

template <int F>
cudaError_t launch_rows(const AcceptParams& p, cudaStream_t st) {
    const size_t smem = rows_smem(p.groups, p.nbuf);
    cudaError_t e = set_rows_attrs<F>(p.C, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.nclusters * p.C, 1, 1);
    cfg.blockDim = dim3(kRT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, accept_rows_kernel<F>, p);
}

template <int F>
cudaError_t max_clusters(int C, size_t smem, int* out) {
    cudaError_t e = set_rows_attrs<F>(C, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C, 1, 1);
    cfg.blockDim = dim3(kRT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(out, accept_rows_kernel<F>, &cfg);
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
        default: return cudaErrorNotSupported;         \
    }

cudaError_t max_clusters_dispatch(int F, int C, size_t smem, int* out) {
    RAPID_ACCEPT_DISPATCH(max_clusters, F, C, smem, out)
}

cudaError_t launch_rows_dispatch(int F, const AcceptParams& p, cudaStream_t st) {
    RAPID_ACCEPT_DISPATCH(launch_rows, F, p, st)
}

AcceptShape shape_for(int V, int C) {
    AcceptShape sh{};
    sh.vocab = V;
    sh.cluster = C;
    sh.chunk = ((V + C - 1) / C + 3) / 4 * 4;
    sh.groups = (sh.chunk / 4 + 31) / 32 * 32;
    sh.F = (sh.groups + kGT - 1) / kGT;
    sh.nbuf = kGroups;   // one resident row per warp group
    return sh;
}

// Co-resident clusters per (device, F, C, shared memory), cached: the
// occupancy query is not free.
struct OccEntry {
    int dev, F, C;
    size_t smem;
    int n;
};
std::mutex g_occ_mu;
OccEntry g_occ[64];
int g_nocc = 0;

int occupancy(int dev, int F, int C, size_t smem) {
    {
        std::lock_guard<std::mutex> lk(g_occ_mu);
        for (int i = 0; i < g_nocc; ++i) {
            const OccEntry& o = g_occ[i];
            if (o.dev == dev && o.F == F && o.C == C && o.smem == smem) return o.n;
        }
    }
    int n = 0;
    if (max_clusters_dispatch(F, C, smem, &n) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    std::lock_guard<std::mutex> lk(g_occ_mu);
    if (g_nocc < 64) g_occ[g_nocc++] = OccEntry{dev, F, C, smem, n};
    return n;
}

}  // namespace

cudaError_t accept_plan(int V, int rows, AcceptShape* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int cmin = (V + kAcceptMaxSlice - 1) / kAcceptMaxSlice;
    if (cmin < 1) cmin = 1;
    int cmax = (V + kMinSlice - 1) / kMinSlice;
    if (cmax > kAcceptMaxCluster) cmax = kAcceptMaxCluster;
    if (cmax < cmin) cmax = cmin;
    bool found = false;
    int64_t best_cost = 0;
    AcceptShape best{};
    for (int C = cmin; C <= cmax && C <= kAcceptMaxCluster; ++C) {
        AcceptShape sh = shape_for(V, C);
        if (sh.F > kAcceptMaxF || rows_smem(sh.groups, sh.nbuf) > kSmemBudget) continue;
        sh.max_clusters = occupancy(dev, sh.F, C, rows_smem(sh.groups, sh.nbuf));
        if (sh.max_clusters <= 0) continue;
        const int ncl = rows < sh.max_clusters ? rows : sh.max_clusters;
        const int64_t cost = (int64_t)((rows + ncl - 1) / ncl) * sh.chunk;
        if (!found || cost < best_cost || (cost == best_cost && sh.nbuf > best.nbuf)) {
            found = true;
            best_cost = cost;
            best = sh;
        }
    }
    if (!found) return cudaErrorNotSupported;
    *out = best;
    return cudaSuccess;
}

cudaError_t launch_accept(const AcceptParams& p0, const AcceptShape& sh, cudaStream_t st) {
    AcceptParams p = p0;
    p.C = sh.cluster;
    p.chunk = sh.chunk;
    p.groups = sh.groups;
    p.nbuf = sh.nbuf;
    p.rows = p.B * p.n_q;
    p.nclusters = p.rows < sh.max_clusters ? p.rows : sh.max_clusters;
    if (p.nclusters < 1 || p.chunk > kAcceptMaxSlice) return cudaErrorNotSupported;
    cudaError_t e = launch_rows_dispatch(sh.F, p, st);
    if (e != cudaSuccess) return e;
    // The selection slices row e on its own: one CTA per kSelSlice entries,
    // at most kAcceptMaxCluster, so that each CTA's share of the re-read is
    // in flight in one round of loads -- while the batch's clusters still fit
    // in one wave (kSelPerSm CTAs per SM); larger batches keep the row
    // kernel's slices (fewer CTAs repeating the path search).
    int sc = (p.V + kSelSlice - 1) / kSelSlice;
    if (sc > kAcceptMaxCluster) sc = kAcceptMaxCluster;
    if (sc < 1) sc = 1;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if ((int64_t)p.B * sc > (int64_t)kSelPerSm * sms) sc = p.C;
    p.C = sc;
    p.chunk = ((p.V + sc - 1) / sc + 3) / 4 * 4;
    if (p.chunk > kAcceptMaxSlice) return cudaErrorNotSupported;
    const size_t sel_smem = (size_t)p.chunk * 4;
    e = cudaFuncSetAttribute(accept_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sel_smem);
    if (e != cudaSuccess) return e;
    if (p.C > 8) {
        e = cudaFuncSetAttribute(accept_select_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.C, p.B, 1);
    cfg.blockDim = dim3(kST, 1, 1);
    cfg.dynamicSmemBytes = sel_smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, accept_select_kernel, p);
}

}  // namespace rapid
