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
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(LmBars) <= 256, "barrier block too small");

// Codes recorded by a timed-out wait: role << 24 | barrier << 16 | step.
enum : unsigned int {
    kLmProducer = 1u << 24, kLmMma = 2u << 24, kLmEpilogue = 3u << 24,
    kLmFull = 1u << 16, kLmEmpty = 2u << 16, kLmAccFull = 3u << 16, kLmAccEmpty = 4u << 16,
    kLmDrain = 5u << 16
};

template <int N>
__global__ void __launch_bounds__(kThreadsLm, 1)
lm_head_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmW64,
               const __grid_constant__ CUtensorMap tmW32, const __grid_constant__ CUtensorMap tmW16,
               const __grid_constant__ CUtensorMap tmH, int rows, int hidden, int V,
               float* __restrict__ z, unsigned int* err) {
    using L = LmPlan<N>;
    constexpr int S = L::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    LmBars* bars = reinterpret_cast<LmBars*>(smem + L::kBarOff);
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

    if (warp == 0) {
        // ------------------------------ TMA producer --------------------------
        if (lane == 0) {
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
                        tma_load_2d(stage, &tmW, kb * kKB, y, &bars->full[st]);
                    } else {
                        // a shorter tile as at most three boxes of 64, 32 and 16
                        // rows, each landing where those rows of a full box would
                        // (whole 1024-byte swizzle atoms: the same layout)
                        int u = 0;
                        if (h & 64) {
                            tma_load_2d(stage, &tmW64, kb * kKB, y, &bars->full[st]);
                            u += 64;
                        }
                        if (h & 32) {
                            tma_load_2d(stage + u * kKB * 2, &tmW32, kb * kKB, y + u, &bars->full[st]);
                            u += 32;
                        }
                        if (h & 16)
                            tma_load_2d(stage + u * kKB * 2, &tmW16, kb * kKB, y + u, &bars->full[st]);
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
    } else {
        // ------------------------------ epilogue ------------------------------
        const int q4 = warp & 3;                       // TMEM lane quadrant
        const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
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
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (c0 + i < rows) z[(int64_t)(c0 + i) * V + v] = __uint_as_float(r[i]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->acc_empty[buf]);
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
    auto kern = lm_head_kernel<N>;
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
    return cudaLaunchKernelEx(&cfg, kern, tmW, tmW64, tmW32, tmW16, tmH, rows, hidden_dim, V, z,
                              err);
}

}  // namespace

bool lm_head_supported() { return tensor_map_encoder() != nullptr; }

cudaError_t launch_lm_head(const void* hidden, const void* W, int rows, int hidden_dim, int V,
                           float* z, unsigned int* err, cudaStream_t st) {
    if (rows <= 16) return launch_n<16>(hidden, W, rows, hidden_dim, V, z, err, st);
    if (rows <= 32) return launch_n<32>(hidden, W, rows, hidden_dim, V, z, err, st);
    if (rows <= 64) return launch_n<64>(hidden, W, rows, hidden_dim, V, z, err, st);
    if (rows <= 128) return launch_n<128>(hidden, W, rows, hidden_dim, V, z, err, st);
    return launch_n<256>(hidden, W, rows, hidden_dim, V, z, err, st);
}

}  // namespace rapid
