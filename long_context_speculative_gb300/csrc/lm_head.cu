// Target logits of the verify rows from their final hidden states and the LM
// head, on the tensor cores (sm_103a).
//
// "LongSpec: Long-Context Lossless Speculative Decoding with Efficient
// Drafting and Verification", section 2.1: the drafter shares the target's
// embedding and LM head; "RAPID: Long-Context Inference with Retrieval-
// Augmented Speculative Decoding", section 2.1: z is the target's logit
// vector over the vocabulary, which the acceptance step consumes.
//
// z = H W^T with a handful of rows (the n_q verify rows of each sequence)
// and the whole vocabulary: a GEMV-shaped product bound by reading W once
// (V x hidden bf16, 1.05 GB for a 128256 x 4096 head).  It runs as a
// tcgen05 product with the operands swapped: A = a 128-entry slice of W
// (M = 128 vocabulary rows, K-major, as stored), B = the hidden states
// (N = rows padded to 16..256, K-major), so each vocabulary tile is one
// M128 x N accumulator in tensor memory and W streams through shared memory
// exactly once.
//
// CTA (persistent, one per SM): a contiguous run of vocabulary rows, cut in
// 16-row units so that every SM gets the same share to within 16 rows
// (whole 128-row tiles would leave the last wave 6 % short of full); the run
// is taken as 128-row tiles, the last one possibly shorter (a multiple of 16
// rows, loaded as up to three smaller boxes; the MMA still computes 128 rows and the rows
// past the run are not stored).  192 threads:
//   warp 0     TMA producer: per 64-wide hidden block, the tile's rows of W
//              (one 128 x 64 box, 16 KB, or boxes of 64, 32, 16 rows) and an
//              N x 64 box of H (rows past the last are zero-filled by the
//              copy) into a ring of up to 12 stages.
//   warp 1     allocates tensor memory and issues the MMAs (one thread):
//              four M128 N K16 products per stage into one of two
//              accumulator buffers, alternating by tile.
//   warps 2-5  epilogue, one per tensor-memory lane quadrant: a finished
//              accumulator is read back (16 columns at a time) and written as
//              z[r][v] for the real rows (32 consecutive v per warp store).
// Every wait is bounded in wall-clock time; on a timeout the kernel records
// an error, stops issuing, drains what it issued and returns.
//
// Fused variant (rapid_lm_head_accept for up to 16 rows): the epilogue keeps
// the CTA's run of z in shared memory instead of writing it, the producer
// copies the same run of q beside it, and after the product the CTA runs the
// acceptance step of "RAPID ...", sections 2.1 and 2.4, on its run: the
// vocabulary-wide (max, sum) of z / T and of the augmented logits, the
// ratio tests, the path choice and the residual (or bonus) draw, with one
// grid-wide barrier after each of the three vocabulary-wide reductions.  The
// launch is cooperative (every CTA resident, one per SM), and every barrier
// wait is bounded like the others.
#include <cuda_bf16.h>

#include "common.cuh"
#include "lm_head.cuh"
#include "tcgen05.cuh"

namespace rapid {

namespace {

constexpr int kVT = 128;                    // vocabulary rows per tile (MMA M)
constexpr int kVU = 16;                     // vocabulary rows per scheduling unit
constexpr int kKB = 64;                     // hidden elements per stage (128 bytes of bf16)
constexpr int kWBytes = kVT * kKB * 2;      // 16 KB of W per stage
constexpr int kThreadsLm = 192;
// The fused variant adds ten warps that wait during the product and give its
// acceptance tail one warp per row (and per sequence).
constexpr int kThreadsFused = 512;
constexpr int kMaxStagesLm = 12;
constexpr int kStageBudget = 216 * 1024;

template <int N>
struct LmPlan {
    static constexpr int kHBytes = N * kKB * 2;
    static constexpr int kStageBytes = kWBytes + kHBytes;
    static constexpr int kStages =
        kStageBudget / kStageBytes < kMaxStagesLm ? kStageBudget / kStageBytes : kMaxStagesLm;
    static constexpr int kBarOff = kStages * kStageBytes;
    static constexpr int kSmemBytes = kBarOff + 256 + 1024;   // + barriers + alignment slack
    static constexpr uint32_t kTmemCols = 2 * N < 32 ? 32 : 2 * N;
    // kind::f16: D = f32, A = B = bf16, both K-major, N / 8 at bit 17, M / 16 at bit 24
    static constexpr uint32_t kIdesc =
        (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(kVT >> 4) << 24);
    static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct LmBars {
    uint64_t full[kMaxStagesLm];
    uint64_t empty[kMaxStagesLm];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint64_t q_full;      // fused variant: this CTA's run of q landed
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(LmBars) <= 256, "barrier block too small");

// Codes recorded by a timed-out wait: role << 24 | barrier << 16 | step.
enum : unsigned int {
    kLmProducer = 1u << 24, kLmMma = 2u << 24, kLmEpilogue = 3u << 24, kLmTail = 4u << 24,
    kLmFull = 1u << 16, kLmEmpty = 2u << 16, kLmAccFull = 3u << 16, kLmAccEmpty = 4u << 16,
    kLmDrain = 5u << 16, kLmQFull = 6u << 16, kLmGrid = 7u << 16
};

// 2^x on the SFU (flushes denormal results to zero, as the acceptance kernels do)
__device__ __forceinline__ float ex2f_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <bool FUSED>
__device__ void accept_tail(const LmAcceptParams& fa, const float* zs, const float* qs, int rows,
                            int V, int v0, int n, unsigned int* err, float2* ring);

template <int N, bool FUSED>
__global__ void __launch_bounds__(FUSED ? kThreadsFused : kThreadsLm, 1)
lm_head_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmW64,
               const __grid_constant__ CUtensorMap tmW32, const __grid_constant__ CUtensorMap tmW16,
               const __grid_constant__ CUtensorMap tmH, int rows, int hidden, int V,
               float* __restrict__ z, unsigned int* err, const LmAcceptParams fa) {
    using L = LmPlan<N>;
    // the fused variant gives part of the ring's shared memory to z and q
    const int S = FUSED ? fa.stages : L::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int bar_off = S * L::kStageBytes;
    LmBars* bars = reinterpret_cast<LmBars*>(smem + bar_off);
    float* zs = reinterpret_cast<float*>(smem + bar_off + 256);   // fused: [rows][run_max]
    float* qs = zs + (FUSED ? (size_t)rows * fa.run_max : 0);
    __shared__ float2 s_ep[4][FUSED ? kLmFusedMaxRows : 1];   // fused: per epilogue warp, per row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this CTA's vocabulary rows [v_begin, v_end), in whole 16-row units
    const int units = (V + kVU - 1) / kVU;
    const int v_begin = (int)((int64_t)units * blockIdx.x / gridDim.x) * kVU;
    const int v_end = (int)((int64_t)units * (blockIdx.x + 1) / gridDim.x) * kVU;
    const int n_tiles = (v_end - v_begin + kVT - 1) / kVT;
    const int kb_n = hidden / kKB;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&bars->full[i], 1);
            mbar_init(&bars->empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->acc_full[i], 1);
            mbar_init(&bars->acc_empty[i], 4);
        }
        mbar_init(&bars->drain, 1);
        mbar_init(&bars->q_full, 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&bars->tmem_base)),
                     "r"(L::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_wait();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t sbase = smem_u32(smem);

    const int v_real = (v_end < V ? v_end : V) - v_begin;   // real vocabulary entries of the run
    if (warp == 0) {
        // ------------------------------ TMA producer --------------------------
        if (lane == 0) {
            if constexpr (FUSED) {
                // this CTA's run of q, every row, beside the ring (16-byte
                // aligned: V % 4 == 0 and v_begin a multiple of 16)
                mbar_arrive_expect_tx(&bars->q_full, (uint32_t)(rows * v_real * 4));
                if (v_real > 0)
                    for (int r = 0; r < rows; ++r)
                        bulk_g2s(qs + (size_t)r * fa.run_max, fa.q + (int64_t)r * V + v_begin,
                                 (uint32_t)(v_real * 4), &bars->q_full);
            }
            // the head is read once: its lines go first when L2 needs room
            const uint64_t w_policy = l2_policy_evict_first();
            int it = 0, issued = 0;
            bool ok = true;
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int y = v_begin + j * kVT;
                const int h = v_end - y < kVT ? v_end - y : kVT;   // rows of this tile, 16 | h
                for (int kb = 0; kb < kb_n; ++kb, ++it) {
                    const int st = it % S;
                    if (it >= S && !mbar_wait_sleep(&bars->empty[st], ((it / S) + 1) & 1, err,
                                                    kLmProducer | kLmEmpty | (unsigned)(it & 0xffff))) {
                        ok = false;
                        break;
                    }
                    if (*((volatile int*)&bars->abort)) {
                        ok = false;
                        break;
                    }
                    uint8_t* stage = smem + st * L::kStageBytes;
                    mbar_arrive_expect_tx(&bars->full[st], (uint32_t)(h * kKB * 2 + L::kHBytes));
                    if (h == kVT) {
                        tma_load_2d_hint(stage, &tmW, kb * kKB, y, &bars->full[st], w_policy);
                    } else {
                        // a shorter tile as at most three boxes of 64, 32 and 16
                        // rows, each landing where those rows of a full box would
                        // (whole 1024-byte swizzle atoms: the same layout)
                        int u = 0;
                        if (h & 64) {
                            tma_load_2d_hint(stage, &tmW64, kb * kKB, y, &bars->full[st], w_policy);
                            u += 64;
                        }
                        if (h & 32) {
                            tma_load_2d_hint(stage + u * kKB * 2, &tmW32, kb * kKB, y + u, &bars->full[st],
                                             w_policy);
                            u += 32;
                        }
                        if (h & 16)
                            tma_load_2d_hint(stage + u * kKB * 2, &tmW16, kb * kKB, y + u, &bars->full[st],
                                             w_policy);
                    }
                    tma_load_2d(stage + kWBytes, &tmH, kb * kKB, 0, &bars->full[st]);
                    ++issued;
                }
            }
            if (!ok) {
                bars->abort = 1;
                // the copies still in flight land before the CTA exits
                for (int i = issued > S ? issued - S : 0; i < issued; ++i)
                    mbar_wait(&bars->full[i % S], (i / S) & 1, nullptr, 0);
            }
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ----------------------------
        if (lane == 0) {
            const uint64_t wd0 = sdesc(sbase, 16, 1024);
            const uint64_t hd0 = sdesc(sbase + kWBytes, 16, 1024);
            int it = 0;
            bool ok = true;
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int buf = j & 1;
                if (j >= 2 && !mbar_wait_sleep(&bars->acc_empty[buf], ((j >> 1) + 1) & 1, err,
                                               kLmMma | kLmAccEmpty | (unsigned)(j & 0xffff))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(buf * N);
                for (int kb = 0; kb < kb_n; ++kb, ++it) {
                    const int st = it % S;
                    if (!mbar_wait_sleep(&bars->full[st], (it / S) & 1, err,
                                         kLmMma | kLmFull | (unsigned)(it & 0xffff)) ||
                        *((volatile int*)&bars->abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t so = (uint64_t)((st * L::kStageBytes) >> 4);
#pragma unroll
                    for (int k = 0; k < kKB / 16; ++k)
                        mma_bf16(d, wd0 + so + (uint64_t)(k * 2), hd0 + so + (uint64_t)(k * 2),
                                 L::kIdesc, (kb > 0 || k > 0) ? 1u : 0u);
                    mma_commit(&bars->empty[st]);
                }
                if (ok) mma_commit(&bars->acc_full[buf]);
            }
            if (!ok) bars->abort = 1;
            // drain: every MMA issued so far has completed once this arrives
            mma_commit(&bars->drain);
            mbar_wait_sleep(&bars->drain, 0, err, kLmMma | kLmDrain);
        }
    } else if (warp < 6) {
        // ------------------------------ epilogue ------------------------------
        const int q4 = warp & 3;                       // TMEM lane quadrant
        const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
        // fused: this lane's running (max, sum of exp(x - max)) of x = z / T
        // per row over its vocabulary entries
        float em[16], es[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            em[i] = -INFINITY;
            es[i] = 0.f;
        }
        for (int j = 0; j < n_tiles; ++j) {
            const int buf = j & 1;
            const bool ok = __all_sync(0xffffffffu,
                                       mbar_wait_sleep(&bars->acc_full[buf], (j >> 1) & 1, err,
                                                       kLmEpilogue | kLmAccFull | (unsigned)(j & 0xffff)));
            if (!ok) {
                if (lane == 0) bars->abort = 1;
                break;
            }
            tc_fence_after();
            const int y = v_begin + j * kVT;
            const int v = y + q4 * 32 + lane;
            const bool mine = v < V && v < v_end;   // rows past the run belong to the next CTA
#pragma unroll 1
            for (int c0 = 0; c0 < N; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(lane_addr + (uint32_t)(buf * N + c0), r);
                tmem_wait_ld();
                if (mine) {
                    if constexpr (FUSED) {
                        float* zv = zs + (v - v_begin);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            if (c0 + i < rows) {
                                const float val = __uint_as_float(r[i]);
                                zv[(size_t)(c0 + i) * fa.run_max] = val;
                                const float x = val * fa.invT;
                                const float mn = fmaxf(em[i], x);
                                es[i] = es[i] * ex2f_approx((em[i] - mn) * kLog2e) +
                                        ex2f_approx((x - mn) * kLog2e);
                                em[i] = mn;
                            }
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (c0 + i < rows) z[(int64_t)(c0 + i) * V + v] = __uint_as_float(r[i]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->acc_empty[buf]);
        }
        if constexpr (FUSED) {
            // the warp's (max, sum) per row, for the CTA's partial of z / T
            for (int i = 0; i < rows; ++i) {
                const float m = warp_max(em[i]);
                const float e = em[i] == -INFINITY ? 0.f : es[i] * ex2f_approx((em[i] - m) * kLog2e);
                const float sum = warp_sum(e);
                if (lane == 0) s_ep[q4][i] = make_float2(m, sum);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(L::kTmemCols)
                     : "memory");
    }
    if constexpr (FUSED) {
        // The run of q has landed (its copy was issued first and is waited
        // for even after an abort, so no copy outlives the CTA).  A CTA whose
        // product gave up still takes part in the barriers, so that the
        // others finish; the error word already marks the outputs invalid.
        if (threadIdx.x == 0) (void)mbar_wait(&bars->q_full, 0u, err, kLmTail | kLmQFull);
        if (threadIdx.x < rows) {   // the CTA's (max, sum) of z / T per row
            float m = -INFINITY;
            for (int w = 0; w < 4; ++w)
                if (s_ep[w][threadIdx.x].y > 0.f) m = fmaxf(m, s_ep[w][threadIdx.x].x);
            float sum = 0.f;
            for (int w = 0; w < 4; ++w) {
                const float2 v = s_ep[w][threadIdx.x];
                if (v.y > 0.f) sum += v.y * ex2f_approx((v.x - m) * kLog2e);
            }
            fa.part1[(size_t)threadIdx.x * gridDim.x + blockIdx.x] = make_float2(m, sum);
        }
        __syncthreads();
        accept_tail<true>(fa, zs, qs, rows, V, v_begin, v_real, err, reinterpret_cast<float2*>(smem));
    }
}


// ---------------------------------------------------------------------------
// Acceptance after the product (fused variant)
// ---------------------------------------------------------------------------

// Grid-wide barrier of a cooperative launch: the CTA's writes before it are
// visible to every CTA after it.  bar[0] counts arrivals over the whole call
// (zeroed before the launch); the k-th barrier is passed once it reaches
// k * gridDim.x.  Thread 0 arrives with a release and polls with acquires,
// bounded in wall-clock time: a CTA that gives up records the barrier and
// carries on, the call's outputs being marked invalid by the error word.
__device__ void grid_sync(unsigned int* bar, unsigned int k, unsigned int* err, unsigned int code) {
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned int target = k * gridDim.x;
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(bar) : "memory");
        const uint64_t t0 = global_timer_ns();
        for (;;) {
            unsigned int v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(bar) : "memory");
            if (v >= target) break;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                if (err) {
                    atomicOr(err, kErrWaitTimeout);
                    atomicCAS(err + 1, 0u, code | 0x80000000u);
                }
                break;
            }
        }
    }
    __syncthreads();
}

__device__ __forceinline__ int fa_node_count(const LmAcceptParams& fa, int b) {
    if (!fa.n_nodes) return fa.n_q;
    const int n = fa.n_nodes[b];
    return n < 1 ? 1 : (n > fa.n_q ? fa.n_q : n);
}

__device__ __forceinline__ int fa_parent(const LmAcceptParams& fa, int b, int i) {
    if (!fa.parent) return i - 1;
    int par = fa.parent[(int64_t)b * fa.n_q + i];
    if (par < 0) par = 0;
    if (par > i - 1) par = i - 1;
    return par;
}

constexpr int kTailWarps = kThreadsFused / 32;   // 16: one per row / sequence
constexpr int kMaxGridJ = 8;                      // partials per lane: grids of up to 256 CTAs
static_assert(kTailWarps >= kLmFusedMaxRows, "one tail warp per row");

// (max, sum of exp(. - max)) over the grid of row r from the CTAs' partials
// part[r * G + cc], in every lane of the calling warp; the loads are
// coalesced and all issued before any is used (one round of L2 latency).
__device__ __forceinline__ float2 combine_row(const float2* part, int r) {
    const int lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const float2* pr = part + (size_t)r * G;
    float2 v[kMaxGridJ];
#pragma unroll
    for (int j = 0; j < kMaxGridJ; ++j) {
        const int cc = lane + 32 * j;
        v[j] = cc < G ? __ldcg(pr + cc) : make_float2(-INFINITY, 0.f);
    }
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < kMaxGridJ; ++j)
        if (v[j].y > 0.f) m = fmaxf(m, v[j].x);
    m = warp_max(m);
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxGridJ; ++j)
        if (v[j].y > 0.f) sum += v[j].y * ex2f_approx((v[j].x - m) * kLog2e);
    return make_float2(m, warp_sum(sum));
}

// A running (max, sum of exp(. - max)) of the thread's values, combined over
// the warp; the same result in every lane.
__device__ __forceinline__ float2 warp_ms_pair(float m, float s) {
    const float mw = warp_max(m);
    const float e = m == -INFINITY ? 0.f : s * ex2f_approx((m - mw) * kLog2e);
    return make_float2(mw, warp_sum(e));
}

// The CTA's run of the acceptance step: z and q of every row for vocabulary
// entries [v0, v0 + n) are in shared memory (row pitch fa.run_max), and the
// run's (max, sum) of z / T per row is in fa.part1.  Every CTA runs this; the
// reductions over the vocabulary combine the CTAs' partials after a grid
// barrier.  Same arithmetic as accept.cu: p = exp(x - m1) / s1 with x = z / T,
// a = x + eta (q - p), p_hat = exp(a - m2) / s2 (m2 = max a, so max p_hat =
// 1 / s2), the tail rule p_hat := p below 0.1 max p_hat, accept iff
// r <= min(1, p_hat(t) / q(t)), and the next token by inverse CDF in token
// order over max(p - p_hat, p - q, 0) (or p).
template <bool FUSED>
__device__ void accept_tail(const LmAcceptParams& fa, const float* zs, const float* qs, int rows,
                            int V, int v0, int n, unsigned int* err, float2* ring) {
    constexpr int kR = kLmFusedMaxRows;
    constexpr int kW = kTailWarps;
    constexpr int kT = kThreadsFused;
    __shared__ float s_m1[kR], s_s1[kR], s_m2[kR], s_s2[kR], s_r[kR];
    __shared__ int s_tok[kR], s_par[kR], s_nn[kR], s_acc[kR];
    __shared__ int s_e[kR], s_resid[kR], s_owner[kR];
    __shared__ float s_tin[kR];
    __shared__ float2 s_w[kW][kR];
    __shared__ float s_scan[kW];
    __shared__ float s_diag[kR][5];
    __shared__ int s_len[kR], s_path[kR];
    // the draw's per-CTA masses, [sequence][CTA], in the ring's shared memory
    // (free once the product is done)
    float2 (*s_p3)[32 * kMaxGridJ] = reinterpret_cast<float2 (*)[32 * kMaxGridJ]>(ring);
    __shared__ int s_pick[2];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, G = gridDim.x;
    const int ld = fa.run_max;
    const int n_q = fa.n_q;
    const float invT = fa.invT, eta = fa.eta;
    uint2 key = make_uint2(fa.seed_lo, fa.seed_hi);
    if (fa.seed_dev) {
        const unsigned long long sd = __ldcg(fa.seed_dev);
        key = make_uint2((uint32_t)(sd & 0xffffffffull), (uint32_t)(sd >> 32));
    }

    // ---- node inputs, the ratio tests' uniforms, and (z, q) at the draft
    // tokens this run holds --------------------------------------------------
    if (tid < fa.B) s_nn[tid] = fa_node_count(fa, tid);
    if (tid < rows) {
        const int b = tid / n_q, i = tid - b * n_q;
        const int tok = fa.tokens[tid];
        const int par = i == 0 ? -1 : fa_parent(fa, b, i);
        s_tok[tid] = tok;
        s_par[tid] = par;
        s_r[tid] = word_uniform(philox4x32_10((uint32_t)i, (uint32_t)b, 0u, 0u, key.x, key.y).w[0]);
        if (i >= 1 && tok >= v0 && tok < v0 + n) {
            const size_t off = (size_t)(b * n_q + par) * ld + (tok - v0);
            fa.zq_tok[tid] = make_float2(zs[off], qs[off]);
        }
    }
    grid_sync(fa.bar, 1u, err, kLmTail | kLmGrid | 1u);

    // ---- global (m1, s1); the run's (max, sum) of the augmented logits ----
    // (one warp per row)
    if (warp < rows) {
        const int r = warp;
        const float2 g1 = combine_row(fa.part1, r);
        if (lane == 0) {
            s_m1[r] = g1.x;
            s_s1[r] = g1.y;
        }
        float2 out = make_float2(-INFINITY, 0.f);
        const int b = r / n_q;
        if (r - b * n_q < s_nn[b]) {   // padding rows: q is not read
            const float* zr = zs + (size_t)r * ld;
            const float* qr = qs + (size_t)r * ld;
            const float m1 = g1.x, is1 = 1.f / g1.y;
            float am = -INFINITY, sum = 0.f;
            if (eta <= 32.f) {
                // a <= x + eta: one reference for every entry, plain sums (two
                // accumulator pairs, so that consecutive entries overlap)
                const float ref = m1 + eta;
                float am2 = -INFINITY, sum2 = 0.f;
                int k = lane;
                for (; k + 32 < n; k += 64) {
                    const float x = zr[k] * invT, x2 = zr[k + 32] * invT;
                    const float pk = ex2f_approx((x - m1) * kLog2e) * is1;
                    const float pk2 = ex2f_approx((x2 - m1) * kLog2e) * is1;
                    const float a = fmaf(eta, qr[k] - pk, x);
                    const float a2 = fmaf(eta, qr[k + 32] - pk2, x2);
                    am = fmaxf(am, a);
                    am2 = fmaxf(am2, a2);
                    sum += ex2f_approx((a - ref) * kLog2e);
                    sum2 += ex2f_approx((a2 - ref) * kLog2e);
                }
                if (k < n) {
                    const float x = zr[k] * invT;
                    const float pk = ex2f_approx((x - m1) * kLog2e) * is1;
                    const float a = fmaf(eta, qr[k] - pk, x);
                    am = fmaxf(am, a);
                    sum += ex2f_approx((a - ref) * kLog2e);
                }
                am = fmaxf(am, am2);
                sum += sum2;
                // relative to this lane's max (sum > 0 whenever that max is
                // within 2 eta of the bound, as the row's maximum always is)
                sum = sum > 0.f ? sum * ex2f_approx((ref - am) * kLog2e) : 0.f;
                if (sum == 0.f) am = -INFINITY;
            } else {
                for (int k = lane; k < n; k += 32) {
                    const float x = zr[k] * invT;
                    const float pk = ex2f_approx((x - m1) * kLog2e) * is1;
                    const float a = fmaf(eta, qr[k] - pk, x);
                    const float mn = fmaxf(am, a);
                    sum = sum * ex2f_approx((am - mn) * kLog2e) + ex2f_approx((a - mn) * kLog2e);
                    am = mn;
                }
            }
            out = warp_ms_pair(am, sum);
            if (!(out.y > 0.f)) out = make_float2(-INFINITY, 0.f);
        }
        if (lane == 0) fa.part2[(size_t)r * G + c] = out;
    }
    grid_sync(fa.bar, 2u, err, kLmTail | kLmGrid | 2u);

    // ---- global (m2, s2); ratio tests; path choice -------------------------
    // (z, q) at every draft token: loaded beside the combine
    const float2 zq = tid < rows ? __ldcg(&fa.zq_tok[tid]) : make_float2(0.f, 0.f);
    if (warp < rows) {
        const float2 g2 = combine_row(fa.part2, warp);
        if (lane == 0) {
            s_m2[warp] = g2.x;   // m2 = max a, so max p_hat = 1 / s2
            s_s2[warp] = g2.y;
        }
    }
    __syncthreads();
    if (tid < rows) {
        const int b = tid / n_q, i = tid - b * n_q;
        int acc = 1;   // the root
        if (i >= 1 && i < s_nn[b]) {
            const int row = b * n_q + s_par[tid];
            const int tok = s_tok[tid];
            acc = 0;
            if (tok >= 0 && tok < V) {
                const float x = zq.x * invT;
                const float pt = ex2f_approx((x - s_m1[row]) * kLog2e) / s_s1[row];
                const float a = fmaf(eta, zq.y - pt, x);
                float ph = ex2f_approx((a - s_m2[row]) * kLog2e) / s_s2[row];
                const float thr = fa.clamp ? 0.1f / s_s2[row] : -1.0f;
                if (ph < thr) ph = pt;
                const float ratio = zq.y == 0.f ? INFINITY : ph / zq.y;
                acc = s_r[tid] <= fminf(1.0f, ratio) ? 1 : 0;
                s_diag[tid][0] = pt; s_diag[tid][1] = ph; s_diag[tid][2] = zq.y;
                s_diag[tid][3] = ratio; s_diag[tid][4] = s_r[tid];
            }
            if (c == 0 && err) {   // device-side inputs out of range (clamped or rejected)
                bool bad = tok < 0 || tok >= V;
                if (fa.parent) {
                    const int par = fa.parent[tid];
                    bad = bad || par < 0 || par >= i;
                }
                if (bad) atomicOr(err, kErrBadInput);
            }
        } else if (i == 0 && c == 0) {
            if (fa.n_nodes && err) {
                const int cnt = fa.n_nodes[b];
                if (cnt < 1 || cnt > n_q) atomicOr(err, kErrBadInput);
            }
        }
        s_acc[tid] = acc;
    }
    __syncthreads();
    if (warp < fa.B) {
        // warp b, lane i = node i: every leaf counts the accepted nodes from
        // the root down its path; the most accepted wins, ties to the
        // smallest leaf id (parents by shuffles, at most n_q steps up)
        const int b = warp, i = lane;
        const int nn = s_nn[b];
        const bool node = i < nn;
        const int par = node ? s_par[b * n_q + i] : 0;
        const unsigned accm = __ballot_sync(0xffffffffu, node && s_acc[b * n_q + i]);
        const unsigned kidm = __reduce_or_sync(0xffffffffu, (node && i > 0) ? (1u << par) : 0u);
        int v = i, depth = 0, top_rej = 0;   // depth of the topmost rejected node on the path
        for (int step = 0; step < n_q; ++step) {
            const int pv = __shfl_sync(0xffffffffu, par, v & 31);
            if (v != 0) {
                ++depth;
                if (!((accm >> v) & 1u)) top_rej = depth;   // overwritten going up: the topmost
                v = pv;
            }
        }
        // len = nodes accepted from the root: above the topmost rejection
        const int len = top_rej == 0 ? depth : depth - top_rej;
        const bool leaf = node && !((kidm >> i) & 1u);
        const int key_l = leaf ? ((len << 8) | (255 - i)) : -1;
        const int best = __reduce_max_sync(0xffffffffu, key_l);
        const int best_len = best >> 8, best_leaf = 255 - (best & 255);
        // the winning leaf's ancestors (and itself), and every node's depth
        int on = 0, w = best_leaf;
        for (int step = 0; step <= n_q; ++step) {
            if (w != 0) on |= 1 << w;
            const int pw = __shfl_sync(0xffffffffu, par, w & 31);
            if (w != 0) w = pw;
        }
        const bool on_path = node && i > 0 && ((on >> i) & 1);
        const int dpt = depth;   // this node's depth below the root
        const unsigned at_e = __ballot_sync(0xffffffffu, on_path && dpt == best_len);
        const int e = best_len > 0 ? __ffs(at_e) - 1 : 0;
        if (lane == 0) {
            s_e[b] = e;
            s_resid[b] = ((kidm >> e) & 1u) ? 1 : 0;
            s_len[b] = best_len;
        }
        if (c == 0) {
            // lane k keeps path[k]: the winning path's node of depth k + 1
            // for k < best_len, else -1 (one ballot per depth, whole warp)
            int val = -1;
            for (int k = 0; k < n_q; ++k) {
                const unsigned m = __ballot_sync(0xffffffffu, on_path && dpt == k + 1);
                if (i == k && k < best_len && m) val = __ffs(m) - 1;
            }
            if (i < n_q) s_path[b * n_q + i] = val;
        }
    }
    __syncthreads();

    // ---- the run's residual (and p) mass of each sequence's row e: thread t
    // takes a contiguous segment of the run; the segments' masses stay in the
    // ring's shared memory for the scan of the CTA that holds the target -----
    const int seg = (n + kT - 1) / kT;
    const int a0 = min(n, tid * seg), a1 = min(n, a0 + seg);
    float2* s_seg = ring + 32 * kMaxGridJ * kR;   // [sequence][thread]: (residual, p) of the segment
    for (int b = 0; b < fa.B; ++b) {
        const int row = b * n_q + s_e[b];
        const float* zr = zs + (size_t)row * ld;
        const float* qr = qs + (size_t)row * ld;
        const float m1 = s_m1[row], is1 = 1.f / s_s1[row];
        const float m2 = s_m2[row], is2 = 1.f / s_s2[row];
        const float thr = fa.clamp ? 0.1f * is2 : -1.0f;
        const bool kids = s_resid[b] != 0;
        float wr = 0.f, wp = 0.f;
        for (int k = a0; k < a1; ++k) {
            const float x = zr[k] * invT;
            const float pk = ex2f_approx((x - m1) * kLog2e) * is1;
            wp += pk;
            if (kids) {
                const float qk = qr[k];
                const float a = fmaf(eta, qk - pk, x);
                float ph = ex2f_approx((a - m2) * kLog2e) * is2;
                if (ph < thr) ph = pk;
                wr += pk - fminf(pk, fminf(ph, qk));   // max(p - p_hat, p - q, 0)
            }
        }
        s_seg[b * kT + tid] = make_float2(wr, wp);
        wr = warp_sum(wr);
        wp = warp_sum(wp);
        if (lane == 0) s_w[warp][b] = make_float2(wr, wp);
    }
    __syncthreads();
    if (tid < fa.B) {
        float2 t = make_float2(0.f, 0.f);
        for (int w = 0; w < kW; ++w) {
            t.x += s_w[w][tid].x;
            t.y += s_w[w][tid].y;
        }
        fa.part3[(size_t)tid * G + c] = t;
    }
    grid_sync(fa.bar, 3u, err, kLmTail | kLmGrid | 3u);

    // ---- the draw: which CTA's run holds each sequence's target ------------
    if (warp < fa.B) {
        const int b = warp;
        const float2* pb = fa.part3 + (size_t)b * G;
#pragma unroll
        for (int j = 0; j < kMaxGridJ; ++j) {   // coalesced, then by lane chunks
            const int cc = lane + 32 * j;
            s_p3[b][cc] = cc < G ? __ldcg(pb + cc) : make_float2(0.f, 0.f);
        }
        __syncwarp();
        const int per = (G + 31) / 32;   // CTAs per lane, in vocabulary order
        float wr = 0.f, wp = 0.f;
        for (int j = 0; j < per; ++j) {
            const float2 v = s_p3[b][lane * per + j];
            wr += v.x;
            wp += v.y;
        }
        const bool resid = s_resid[b] != 0 && warp_sum(wr) > 0.f;   // else p
        const float mine = resid ? wr : wp;
        float incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const float total = __shfl_sync(0xffffffffu, incl, 31);
        const Philox4 rnd = philox4x32_10((uint32_t)(s_e[b] + 1), (uint32_t)b, 0u, 0u, key.x, key.y);
        const float target = word_uniform(rnd.w[1]) * total;
        const unsigned hit = __ballot_sync(0xffffffffu, mine > 0.f && incl > target);
        const unsigned pos = __ballot_sync(0xffffffffu, mine > 0.f);
        int lsel = -1;
        if (hit) lsel = __ffs(hit) - 1;
        else if (pos) lsel = 31 - __clz(pos);   // rounding left the target past the end
        int owner = -1;
        float tin = INFINITY;
        if (lane == lsel) {
            float acc = incl - mine;
            int last = -1;
            for (int j = 0; j < per; ++j) {
                const int cc = lane * per + j;
                const float w = resid ? s_p3[b][cc].x : s_p3[b][cc].y;
                if (w > 0.f) {
                    last = cc;
                    if (acc + w > target) {
                        owner = cc;
                        tin = target - acc;
                        break;
                    }
                }
                acc += w;
            }
            if (owner < 0) owner = last;
        }
        if (lsel >= 0) {
            owner = __shfl_sync(0xffffffffu, owner, lsel);
            tin = __shfl_sync(0xffffffffu, tin, lsel);
        }
        if (lane == 0) {
            s_owner[b] = owner;   // -1: no mass at all (degenerate input)
            s_tin[b] = tin;
            s_resid[b] = resid ? 1 : 0;
            if (owner < 0 && c == 0) fa.next_token[b] = 0;
        }
    }
    __syncthreads();
    if (c == 0) {   // outputs (off the critical path: after the last barrier)
        if (tid < fa.B) fa.n_accepted[tid] = s_len[tid];
        if (tid < rows) {
            const int b = tid / n_q, i = tid - b * n_q;
            if (fa.path) fa.path[tid] = s_path[tid];
            if (fa.diag && (i == 0 || i < s_nn[b])) {
                float* dg = fa.diag + (size_t)tid * 5;
                const bool real = i >= 1 && s_tok[tid] >= 0 && s_tok[tid] < V;
                for (int k = 0; k < 5; ++k)
                    if (i == 0) dg[k] = 0.f;
                    else if (real) dg[k] = s_diag[tid][k];
            }
        }
    }
    // the owner's run: warp 0 finds the segment whose running sum passes the
    // target (lane l holds segments 16 l .. 16 l + 15), and the thread of that
    // segment scans it
    constexpr int kSegPerLane = kT / 32;
    for (int b = 0; b < fa.B; ++b) {
        if (s_owner[b] != c) continue;   // the same in every thread
        const bool resid = s_resid[b] != 0;
        const float tin = s_tin[b];
        if (warp == 0) {
            float ls[kSegPerLane];
            float lsum = 0.f;
#pragma unroll
            for (int j = 0; j < kSegPerLane; ++j) {
                const float2 sg = s_seg[b * kT + lane * kSegPerLane + j];
                ls[j] = resid ? sg.x : sg.y;
                lsum += ls[j];
            }
            float incl = lsum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, lsum > 0.f && incl > tin);
            const unsigned pos = __ballot_sync(0xffffffffu, lsum > 0.f);
            int ln = -1;
            if (hit) ln = __ffs(hit) - 1;
            else if (pos) ln = 31 - __clz(pos);
            int pick = -1;
            float before = 0.f;
            if (lane == ln) {
                // (fully unrolled, so ls stays in registers)
                float acc = incl - lsum, acc_last = acc;
                int last = -1;
#pragma unroll
                for (int j = 0; j < kSegPerLane; ++j) {
                    if (pick < 0 && ls[j] > 0.f) {
                        last = lane * kSegPerLane + j;
                        acc_last = acc;
                        if (acc + ls[j] > tin) {
                            pick = lane * kSegPerLane + j;
                            before = acc;
                        }
                    }
                    if (pick < 0) acc += ls[j];
                }
                if (pick < 0) {
                    pick = last;
                    before = acc_last;
                }
            }
            if (ln >= 0) {
                pick = __shfl_sync(0xffffffffu, pick, ln);
                before = __shfl_sync(0xffffffffu, before, ln);
            }
            if (lane == 0) {
                s_pick[0] = pick;
                s_scan[0] = before;
            }
        }
        __syncthreads();
        const int pick = s_pick[0];
        if (pick < 0) {   // the owner's run has no mass (rounding): its first entry
            if (tid == 0) fa.next_token[b] = v0;
        } else if (tid == pick) {
            const int row = b * n_q + s_e[b];
            const float* zr = zs + (size_t)row * ld;
            const float* qr = qs + (size_t)row * ld;
            const float m1 = s_m1[row], is1 = 1.f / s_s1[row];
            const float m2 = s_m2[row], is2 = 1.f / s_s2[row];
            const float thr = fa.clamp ? 0.1f * is2 : -1.0f;
            float ce = s_scan[0];
            int kpick = -1, klast = -1;
            for (int k = a0; k < a1; ++k) {
                const float x = zr[k] * invT;
                const float pk = ex2f_approx((x - m1) * kLog2e) * is1;
                float w = pk;
                if (resid) {
                    const float qk = qr[k];
                    const float a = fmaf(eta, qk - pk, x);
                    float ph = ex2f_approx((a - m2) * kLog2e) * is2;
                    if (ph < thr) ph = pk;
                    w = pk - fminf(pk, fminf(ph, qk));
                }
                if (w > 0.f) {
                    klast = k;
                    if (ce + w > tin) {
                        kpick = k;
                        break;
                    }
                }
                ce += w;
            }
            if (kpick < 0) kpick = klast;
            fa.next_token[b] = v0 + kpick;
        }
        __syncthreads();
    }
}

// 2-D bf16 view [outer, inner] with an (inner 64) x (box_outer) box, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
              uint32_t box_outer) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
    cuuint32_t box[2] = {(cuuint32_t)kKB, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count_lm() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            n = 1;
    }
    return n;
}

template <int N>
cudaError_t launch_n(const void* hidden, const void* W, int rows, int hidden_dim, int V, float* z,
                     unsigned int* err, cudaStream_t st) {
    CUtensorMap tmW, tmW64, tmW32, tmW16, tmH;
    if (!make_map(&tmW, W, (uint64_t)hidden_dim, (uint64_t)V, kVT) ||
        !make_map(&tmW64, W, (uint64_t)hidden_dim, (uint64_t)V, 64) ||
        !make_map(&tmW32, W, (uint64_t)hidden_dim, (uint64_t)V, 32) ||
        !make_map(&tmW16, W, (uint64_t)hidden_dim, (uint64_t)V, kVU) ||
        !make_map(&tmH, hidden, (uint64_t)hidden_dim, (uint64_t)rows, N))
        return cudaErrorInvalidValue;
    auto kern = lm_head_kernel<N, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         LmPlan<N>::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int units = (V + kVU - 1) / kVU;
    const int sms = sm_count_lm();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(units < sms ? units : sms, 1, 1);
    cfg.blockDim = dim3(kThreadsLm, 1, 1);
    cfg.dynamicSmemBytes = LmPlan<N>::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const LmAcceptParams none{};
    return cudaLaunchKernelEx(&cfg, kern, tmW, tmW64, tmW32, tmW16, tmH, rows, hidden_dim, V, z,
                              err, none);
}

int coop_supported() {
    static int v = -1;
    if (v < 0) {
        int dev = 0, a = 0;
        v = (cudaGetDevice(&dev) == cudaSuccess &&
             cudaDeviceGetAttribute(&a, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && a)
                ? 1
                : 0;
    }
    return v;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

bool lm_head_supported() { return tensor_map_encoder() != nullptr; }

size_t lm_accept_scratch_bytes(int grid, int rows, int B) {
    return 256 + align256((size_t)grid * rows * sizeof(float2)) +
           align256((size_t)grid * rows * sizeof(float2)) +
           align256((size_t)grid * B * sizeof(float2)) + align256((size_t)rows * sizeof(float2));
}

cudaError_t launch_lm_head_accept(const void* hidden, const void* W, int hidden_dim, int V,
                                  LmAcceptParams fa, void* scratch, size_t scratch_bytes,
                                  unsigned int* err, cudaStream_t st) {
    constexpr int N = 16;
    using L = LmPlan<N>;
    const int rows = fa.B * fa.n_q;
    if (rows < 1 || rows > kLmFusedMaxRows || (V % 4) != 0 ||
        (reinterpret_cast<uintptr_t>(fa.q) & 15u) || !coop_supported())
        return cudaErrorNotSupported;
    const int units = (V + kVU - 1) / kVU;
    const int sms = sm_count_lm();
    const int grid = units < sms ? units : sms;
    if (grid > 32 * 8) return cudaErrorNotSupported;   // the tail's partial loads: 8 per lane
    fa.run_max = (units + grid - 1) / grid * kVU;
    if (scratch_bytes < lm_accept_scratch_bytes(grid, rows, fa.B)) return cudaErrorNotSupported;
    auto kern = lm_head_kernel<N, true>;
    cudaFuncAttributes fattr;
    cudaError_t e = cudaFuncGetAttributes(&fattr, kern);
    if (e != cudaSuccess) return e;
    // shared memory: the ring, the barrier block, z and q of the run (every
    // row), alignment slack, beside the kernel's static arrays
    const size_t zq = (size_t)2 * rows * fa.run_max * sizeof(float);
    const size_t fixed = 256 + zq + 1024 + fattr.sharedSizeBytes;
    if (fixed >= 232448) return cudaErrorNotSupported;
    int stages = (int)((232448 - fixed) / L::kStageBytes);
    if (stages > kMaxStagesLm) stages = kMaxStagesLm;
    if (stages < 4) return cudaErrorNotSupported;
    // the tail keeps its per-CTA masses (16 x 256 float2) and the segment
    // masses of the draw (16 x 512 float2) in the ring's space
    if ((size_t)stages * L::kStageBytes <
        (size_t)kLmFusedMaxRows * (256 + kThreadsFused) * sizeof(float2))
        return cudaErrorNotSupported;
    fa.stages = stages;
    const size_t smem = (size_t)stages * L::kStageBytes + 256 + zq + 1024;
    CUtensorMap tmW, tmW64, tmW32, tmW16, tmH;
    if (!make_map(&tmW, W, (uint64_t)hidden_dim, (uint64_t)V, kVT) ||
        !make_map(&tmW64, W, (uint64_t)hidden_dim, (uint64_t)V, 64) ||
        !make_map(&tmW32, W, (uint64_t)hidden_dim, (uint64_t)V, 32) ||
        !make_map(&tmW16, W, (uint64_t)hidden_dim, (uint64_t)V, kVU) ||
        !make_map(&tmH, hidden, (uint64_t)hidden_dim, (uint64_t)rows, N))
        return cudaErrorInvalidValue;
    // scratch: barrier words, then the three partial arrays and the token values
    char* ws = static_cast<char*>(scratch);
    fa.bar = reinterpret_cast<unsigned int*>(ws);
    ws += 256;
    fa.part1 = reinterpret_cast<float2*>(ws);
    ws += align256((size_t)grid * rows * sizeof(float2));
    fa.part2 = reinterpret_cast<float2*>(ws);
    ws += align256((size_t)grid * rows * sizeof(float2));
    fa.part3 = reinterpret_cast<float2*>(ws);
    ws += align256((size_t)grid * fa.B * sizeof(float2));
    fa.zq_tok = reinterpret_cast<float2*>(ws);
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreadsFused, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorNotSupported;
    e = cudaMemsetAsync(fa.bar, 0, sizeof(unsigned int), st);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreadsFused, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // the grid barriers need every CTA resident
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmW, tmW64, tmW32, tmW16, tmH, rows, hidden_dim, V,
                              (float*)nullptr, err, fa);
}

cudaError_t launch_lm_head(const void* hidden, const void* W, int rows, int hidden_dim, int V,
                           float* z, unsigned int* err, cudaStream_t st) {
    if (rows <= 16) return launch_n<16>(hidden, W, rows, hidden_dim, V, z, err, st);
    if (rows <= 32) return launch_n<32>(hidden, W, rows, hidden_dim, V, z, err, st);
    if (rows <= 64) return launch_n<64>(hidden, W, rows, hidden_dim, V, z, err, st);
    if (rows <= 128) return launch_n<128>(hidden, W, rows, hidden_dim, V, z, err, st);
    return launch_n<256>(hidden, W, rows, hidden_dim, V, z, err, st);
}

}  // namespace rapid
