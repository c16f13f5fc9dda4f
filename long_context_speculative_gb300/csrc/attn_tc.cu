// Tensor-core history kernel of verify attention (bf16, head_dim 64 or 128,
// up to 512 query rows per KV-head group), written for sm_103a: TMA-staged
// K/V tiles, tcgen05 MMAs with accumulators in tensor memory, warp-specialised.
//
// Hybrid tree attention ("LongSpec: Long-Context Lossless Speculative
// Decoding with Efficient Drafting and Verification", section 2.3) needs no
// mask over the history rows: every query of the group sees every history
// row, so the history pass is a plain split-KV flash-decoding pass.  The GQA
// group's G * n_q query rows form the M = 128 operand of one tcgen05 MMA, so
// every K/V byte is read from HBM once per group.
//
// CTA = (split s, sequence b * Hkv + KV head g); 384 threads:
//   warps 0-7  softmax, in two consumer groups (warps 0-3 take the even
//              tiles of the split, warps 4-7 the odd ones; in a 256-row CTA
//              they are its two 128-row blocks and both take every tile);
//              warp w owns TMEM lane quadrant w % 4, i.e. rows 32 (w % 4) ..
//              + 31 of its group's M = 128 operand.  A
//              group turns its S tile into P (bf16, its own shared buffer;
//              two per block in a 256-row CTA), keeps its running max / sum
//              and rescales its O in TMEM when the max grows by more than 2^8.
//              At the end the two groups combine their (O, m, l) into the
//              split's one partial (a 256-row CTA's blocks write their own).
//   warp 8     TMA producer: 64-key K and V tiles into a ring of 32 KB (16 KB
//              at d = 64) stages filling the shared memory left; the last
//              split also loads the n_q speculative rows as one more tile,
//              which the softmax masks with the chain / tree mask.
//   warp 11    allocates TMEM and issues the MMAs (one thread), in the order
//              their inputs become ready: S_j = Q K_j^T (M128 N64 K = d, two S
//              buffers per group, so S runs a tile ahead of the softmax; in a
//              256-row CTA one per block, released as soon as it is loaded,
//              with Q in TMEM) and O_g += P_i V_i (M128 N = d K64).  It sits
//              on sub-partition 3, whose softmax warps are the most often
//              idle: issue slots taken there slow the tensor pipe's intake.
// Shared-memory operands use the 128-byte swizzle; Q, K and P are K-major,
// V is MN-major (d contiguous).  Every mbarrier wait is bounded in wall-clock
// time; on a timeout the kernel records an error code, stops issuing work,
// drains what it issued and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "attn.cuh"
#include "common.cuh"
#include "tcgen05.cuh"

namespace rapid {

namespace {

constexpr int kSoftmaxWarps = 8;                // two groups x four TMEM lane quadrants
// Warp w runs on SM sub-partition w % 4, and the MMA issuer gets its issue
// slots only between those of the softmax warps on its sub-partition: two busy
// softmax warps beside it slow the tensor pipe's work by a quarter.  So the
// issuer is warp 11, on the sub-partition of TMEM lane quadrant 3 (group rows
// 96..127), whose softmax warps are most often idle: padding rows of a 224-row
// tree group's second block, of an 88-row group, and absent below 97 rows.
// The producer runs on sub-partition 0 (warp 8); warps 9 and 10 are idle.
constexpr int kProducerWarp = kSoftmaxWarps;
constexpr int kMmaWarp = kSoftmaxWarps + 3;
constexpr int kThreads = 32 * (kSoftmaxWarps + 4);
constexpr int kKeys = 64;                       // keys per K/V tile
constexpr int kBlockBytes = kKeys * 128;        // one 64-column block of a K or V tile (8 KB)
constexpr int kMaxStages = 12;
// TMEM columns: S of group g, buffer u at 64 (2 g + u); O of group g at 256 + D g.
// In a 256-row CTA S is single-buffered (block g at 64 g) and Q sits at 128
// (block g at 128 + D g / 2).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemQ = 128;
constexpr uint32_t kTmemO = 256;
constexpr int kBarBytes = 512;

// Shared-memory plan for ROWS query rows kept on chip (64 when the group has
// at most 64 rows, 128 when it has at most 128, else 256) and head dimension D
// (64 or 128).  The MMAs always run with M = 128: with ROWS = 64 the operand
// rows 64..127 of Q and P read the neighbouring shared data and only produce
// output rows that are never used, which frees room for more K/V stages.
// With ROWS = 256 the two consumer groups are the two 128-row blocks of the
// CTA, and each takes every tile: a K/V tile copied into the SM then serves
// 256 query rows instead of 128, which halves the bytes an SM has to take in
// per row of work (the copies in flight, not the HBM bandwidth, bound a CTA
// that runs 128 rows per tile).  The ring takes what shared memory is left:
// 6 / 5 / 4 stages of 32 KB at D = 128, 12 / 11 / 10 stages of 16 KB at D = 64.
template <int ROWS, int D>
struct Plan {
    static constexpr int kD = D;
    static constexpr bool kRowGroups = ROWS > 128;       // groups = row blocks, not even / odd tiles
    static constexpr int kCtaRows = kRowGroups ? 256 : 128;   // group rows one CTA covers
    static constexpr int kGroupRows = kRowGroups ? 128 : ROWS;
    static constexpr int kDBlocks = D / 64;              // 64-column blocks of Q, K and V
    static constexpr int kTileBytes = kKeys * D * 2;     // one K or V tile
    static constexpr int kStageBytes = 2 * kTileBytes;   // K + V
    static constexpr int kActiveQuadrants = kGroupRows / 32;   // softmax warps per group
    static constexpr int kGroupThreads = 32 * kActiveQuadrants;
    static constexpr int kQBlock = ROWS * 128;           // one 64-column block of Q
    static constexpr int kPBytes = kGroupRows * 128;     // one P buffer (64 keys)
    // A 256-row CTA keeps Q in tensor memory (the S products then read only K
    // from shared memory) and double-buffers each block's P in the room that frees.
    static constexpr int kPBufs = kRowGroups ? 4 : 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffP = kOffQ + (kRowGroups ? 0 : kDBlocks * kQBlock);
    static constexpr int kOffKV = kOffP + kPBufs * kPBytes;
    static constexpr int kFit = (232448 - 1024 - kBarBytes - kOffKV) / kStageBytes;
    static constexpr int kStages = kFit < kMaxStages ? kFit : kMaxStages;
    static constexpr int kOffBar = kOffKV + kStages * kStageBytes;
    static constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;   // + 1 KB alignment slack
    // instruction descriptor of O += P V (V MN-major, N = D)
    static constexpr uint32_t kIdescPV = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                                         ((uint32_t)(D >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    static_assert(D == 64 || D == 128, "head dimension 64 or 128");
    static_assert(ROWS == 64 || ROWS == 128 || ROWS == 256, "64, 128 or 256 rows");
    static_assert(kStages >= 4, "too few stages");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Instruction descriptors (kind::f16): D = f32 (bits 4-5 = 1), A = B = bf16
// (bits 7-9 = 1, bits 10-12 = 1), bit 15/16 = A/B MN-major, bits 17-22 = N/8,
// bits 24-28 = M/16.
constexpr uint32_t kIdescS = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kKeys >> 3) << 17) |
                             ((uint32_t)(128 >> 4) << 24);

// 2^x with the SFU instruction (flushes denormal results to zero; P is
// rounded to bf16 afterwards and the running sums tolerate the 2-ulp error).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// A softmax warp's wait.  Groups of at most 64 rows have live warps on
// sub-partitions 0 and 1 only, where polling takes no issue slots from the
// MMA issuer (sub-partition 3) and reacts sooner than a suspended wait: at
// D = 128 that is measurably faster, at D = 64 (tiles turning over twice as
// often, the polls competing with the live warps' own work) it is not.
// Wider groups share the issuer's sub-partition and suspend between polls.
template <bool Poll>
__device__ __forceinline__ bool softmax_wait(uint64_t* bar, uint32_t parity, unsigned int* err,
                                             unsigned int code) {
    if constexpr (Poll) return mbar_wait(bar, parity, err, code);
    else return mbar_wait_sleep(bar, parity, err, code);
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Codes recorded by a timed-out wait: role << 24 | barrier << 16 | tile.
enum : unsigned int {
    kRoleProducer = 1u << 24, kRoleMma = 2u << 24, kRoleSoftmax = 3u << 24,
    kBarKvFull = 1u << 16, kBarKvEmpty = 2u << 16, kBarSFull = 3u << 16,
    kBarPFull = 4u << 16, kBarPFree = 5u << 16, kBarDrain = 6u << 16
};

struct Bars {
    uint64_t kv_full[kMaxStages];
    uint64_t kv_empty[kMaxStages];
    uint64_t s_full[4];   // S buffer u of consumer group g written: index 2 g + u (256 rows: g)
    uint64_t s_free[2];   // 256 rows: block g's S loaded by its softmax warps (one arrival per warp)
    // P of group g written (one arrival per active softmax thread); 256 rows:
    // P buffer 2 g + u of block g written, so that a barrier's next phase (two
    // tiles on) cannot complete before the MMA issuer has seen this one
    uint64_t p_full[4];
    uint64_t p_free[4];   // PV product of group g done (256 rows: of block g from P buffer 2 g + u)
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int grp_ok[2];        // cleared by a group that failed a wait
    SplitOf split;        // this CTA's (sequence, split), computed once by thread 0
};
static_assert(sizeof(Bars) <= kBarBytes, "barrier block too small");

template <int ROWS, int D>
__global__ void __launch_bounds__(kThreads, 1)
attn_prefix_tc_kernel(const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    using L = Plan<ROWS, D>;
    constexpr int kD = L::kD;
    constexpr int kTileBytes = L::kTileBytes;
    constexpr int kStageBytes = L::kStageBytes;
    constexpr int kStages = L::kStages;
    constexpr int kOffQ = L::kOffQ;
    constexpr int kOffP = L::kOffP;
    constexpr int kOffKV = L::kOffKV;
    constexpr int kOffBar = L::kOffBar;
    constexpr int kPBytes = L::kPBytes;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment of the shared-window address (128-byte swizzle atoms).
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    // blockIdx.x = (sequence, split) slot * row_blocks + row block, blockIdx.y
    // = KV head.  The row blocks of one split are adjacent CTAs, so they
    // stream the same K/V tiles together and the second read of each tile is
    // served from L2.  Which (sequence, split) a slot holds is decided on the
    // device from the prefix lengths (split_of), after griddep_wait().
    const int n_rb = tc_row_blocks(p.R);
    const int slot_idx = blockIdx.x / n_rb;
    const int rb = blockIdx.x - slot_idx * n_rb;
    const int r0 = rb * L::kCtaRows;               // first group row of this CTA
    const int Rb = min(L::kCtaRows, p.R - r0);     // rows of this CTA
    const int g = blockIdx.y;
    // The lane quadrants of consumer group gr that hold rows of this CTA: their
    // softmax warps take part, the others leave at once (a group without rows
    // keeps one warp, which runs the barrier protocol alone).
    auto live_quadrants = [&](int gr) -> int {
        const int rows = L::kRowGroups ? Rb - 128 * gr : Rb;
        const int q = (rows + 31) / 32;
        return q < 1 ? 1 : (q > L::kActiveQuadrants ? L::kActiveQuadrants : q);
    };
    // Input-free set-up first: it may overlap the previous kernel in the stream.
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&bars->kv_full[i], 1);
            mbar_init(&bars->kv_empty[i], 1);
        }
        for (int u = 0; u < 4; ++u) mbar_init(&bars->s_full[u], 1);
        for (int gr = 0; gr < 2; ++gr) mbar_init(&bars->s_free[gr], live_quadrants(gr));
        for (int u = 0; u < 4; ++u) {
            // p_full[2 g + u] of block g in a 256-row CTA, p_full[g] otherwise
            mbar_init(&bars->p_full[u], 32 * live_quadrants(L::kRowGroups ? (u >> 1) : (u & 1)));
            mbar_init(&bars->p_free[u], 1);
        }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        bars->grp_ok[0] = 1;
        bars->grp_ok[1] = 1;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&bars->tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    griddep_wait();
    if (tid == 0) {
        const SplitOf sp0 = split_of(p, p.S, slot_idx);
        bars->split = sp0;
        // the merge kernel reads where the partials of this (b, g) are here
        if (sp0.b >= 0 && sp0.s == 0 && rb == 0) {
            p.part_nsplit[sp0.b * p.Hkv + g] = sp0.S_b;
            p.part_first[sp0.b * p.Hkv + g] = slot_idx;
        }
    }
    tc_fence_before();   // the TMEM allocation above, before its address is read
    __syncthreads();
    tc_fence_after();

    // Tiles of this split: the history [0, P) of sequence b in 64-key tiles,
    // shared out evenly over its S_b splits; the last split also takes the n_q
    // speculative rows [P, P + n_q) as one more, masked, tile.
    const SplitOf sp = bars->split;
    const bool has_work = sp.b >= 0;
    const int b = has_work ? sp.b : 0;
    const int s = sp.s;
    const int bg = b * p.Hkv + g;
    const int64_t P = clamped_prefix(p, b);
    const int n_all = sp.tiles;
    const int t_begin = has_work ? (int)(((int64_t)s * n_all) / sp.S_b) : 0;
    const int t_end = has_work ? (int)(((int64_t)(s + 1) * n_all) / sp.S_b) : 0;
    const int n_hist = t_end - t_begin;
    const bool spec_here = has_work && (s == sp.S_b - 1);
    const int n = has_work ? n_hist + (spec_here ? 1 : 0) : 0;
    const int64_t slot = ((int64_t)g * p.nparts + slot_idx) * p.R;   // this CTA's partial rows

    if constexpr (L::kRowGroups) {
        // Q rows of the CTA into tensor memory: softmax warp w writes the rows
        // of its lane quadrant of block w / 4 (K-major, two elements per
        // column); rows >= R are zero.
        if (warp < kSoftmaxWarps && n > 0) {
            const int q4 = warp & 3, gr = warp >> 2;
            const int rr = gr * 128 + q4 * 32 + lane;
            const uint4* src = nullptr;
            if (rr < Rb)
                src = reinterpret_cast<const uint4*>(
                    static_cast<const __nv_bfloat16*>(p.Q) +
                    (((int64_t)b * p.Hq + (int64_t)g * p.G) * p.n_q + r0 + rr) * kD);
            const uint32_t qaddr = bars->tmem_base + ((uint32_t)(q4 * 32) << 16) + kTmemQ +
                                   (uint32_t)(gr * (kD / 2));
#pragma unroll
            for (int h = 0; h < kD / 64; ++h) {   // 64 elements = 32 columns at a time
                uint32_t w[32];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint4 v = src ? src[h * 8 + j] : make_uint4(0, 0, 0, 0);
                    w[4 * j] = v.x; w[4 * j + 1] = v.y; w[4 * j + 2] = v.z; w[4 * j + 3] = v.w;
                }
                tmem_st32(qaddr + (uint32_t)(32 * h), w);
            }
            tmem_wait_st();
        }
    } else if (tid < ROWS && n > 0) {
        // Q rows of the group into shared memory (K-major, 128-byte swizzle);
        // rows >= R are zero.
        const int r = tid;
        constexpr int kQChunks = kD / 8;   // 16-byte pieces of a Q row
        uint4 chunk[kQChunks];
        if (r < Rb) {
            const uint4* src = reinterpret_cast<const uint4*>(
                static_cast<const __nv_bfloat16*>(p.Q) +
                (((int64_t)b * p.Hq + (int64_t)g * p.G) * p.n_q + r0 + r) * kD);
#pragma unroll
            for (int j = 0; j < kQChunks; ++j) chunk[j] = src[j];
        } else {
#pragma unroll
            for (int j = 0; j < kQChunks; ++j) chunk[j] = make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < kQChunks; ++j) {
            const int blk = j >> 3, jj = j & 7;
            *reinterpret_cast<uint4*>(smem + kOffQ + blk * L::kQBlock + r * 128 +
                                      ((jj ^ (r & 7)) << 4)) = chunk[j];
        }
        fence_proxy_async_smem();
    }
    if (has_work && n <= 0 && tid < Rb) {   // empty split: m = -inf, l = 0
        p.part_ml[(slot + r0 + tid) * 2 + 0] = -INFINITY;
        p.part_ml[(slot + r0 + tid) * 2 + 1] = 0.f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t smem_base = smem_u32(smem);
    const int64_t head_row0 = (int64_t)bg * p.cap;

    if (n <= 0) {
        // nothing else to do
    } else if (warp == kProducerWarp) {
        // ------------------------------ TMA producer --------------------------
        if (lane == 0) {
            // A K/V tile read by one CTA only is dead after its copy: with a
            // single row block its L2 lines go first when L2 needs room, so
            // the stream does not push out the partials and code that the
            // merge and the next launches reuse.  Wider groups keep the
            // default policy: the second row block re-reads each tile from L2.
            const uint64_t kv_policy = l2_policy_evict_first();
            const bool once = n_rb == 1;
            // Tile i's rows in the cache (the speculative tile starts at P).
            auto tile_y = [&](int i) -> int {
                const int64_t row0 = (i < n_hist) ? (int64_t)(t_begin + i) * kKeys : P;
                return (int)(head_row0 + row0);
            };
            int issued = 0;
            for (int i = 0; i < n; ++i) {
                const int st = i % kStages;
                if (i >= kStages &&
                    !mbar_wait_sleep(&bars->kv_empty[st], ((i / kStages) + 1) & 1, p.err,
                                     kRoleProducer | kBarKvEmpty | (unsigned)(i & 0xffff))) {
                    bars->abort = 1;
                    break;
                }
                if (*((volatile int*)&bars->abort)) break;
                ++issued;
                uint8_t* kt = smem + kOffKV + st * kStageBytes;
                uint8_t* vt = kt + kTileBytes;
                const int y = tile_y(i);
                mbar_arrive_expect_tx(&bars->kv_full[st], kStageBytes);
#pragma unroll
                for (int c = 0; c < L::kDBlocks; ++c) {   // 64-column blocks of K, then V
                    if (once) {
                        tma_load_2d_hint(kt + c * kBlockBytes, &tmK, 64 * c, y, &bars->kv_full[st],
                                         kv_policy);
                        tma_load_2d_hint(vt + c * kBlockBytes, &tmV, 64 * c, y, &bars->kv_full[st],
                                         kv_policy);
                    } else {
                        tma_load_2d(kt + c * kBlockBytes, &tmK, 64 * c, y, &bars->kv_full[st]);
                        tma_load_2d(vt + c * kBlockBytes, &tmV, 64 * c, y, &bars->kv_full[st]);
                    }
                }
            }
            if (*((volatile int*)&bars->abort)) {
                // let the copies still in flight land before the CTA exits
                for (int i = max(0, issued - kStages); i < issued; ++i)
                    mbar_wait(&bars->kv_full[i % kStages], (i / kStages) & 1, p.err,
                              kRoleProducer | kBarKvFull | (unsigned)(i & 0xffff));
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------ MMA issuer ----------------------------
        // Issues S_j = Q K_j^T and O += P_i V_i in the order their inputs
        // become ready (one loop per configuration below).
        if (lane == 0) {
            // Descriptors are built once; the one of a later operand block is
            // the base plus its byte offset in 16-byte units (all shared
            // addresses stay below 256 KB, so the 14-bit field never carries).
            const uint64_t qd0 = sdesc(smem_base + kOffQ, 16, 1024);
            const uint64_t kd0 = sdesc(smem_base + kOffKV, 16, 1024);
            const uint64_t pd0 = sdesc(smem_base + kOffP, 16, 1024);
            const uint64_t vd0 = sdesc(smem_base + kOffKV + kTileBytes, kBlockBytes, 1024);
            bool ok = true;
            uint64_t t_last = global_timer_ns();
            if constexpr (L::kRowGroups) {
                // The two row blocks move through the tiles together, their
                // products issued in pairs.  S_j (A = Q from tensor memory)
                // goes to the block's one S buffer once its softmax warps
                // have loaded S_{j-1}; PV_i reads P buffer i & 1 of the
                // block; tile i's ring slot is released after its PV pair.
                int ns = 0, npv = 0;
                while (npv < n) {
                    bool progressed = false;
                    // S before PV: the softmax warps wait on S_j now, while
                    // PV_{j-2} is needed only when they write P_j at the
                    // end of the tile.
                    if (ns < n &&
                        (ns == 0 || (mbar_try_wait(&bars->s_free[0], (ns - 1) & 1) &&
                                     mbar_try_wait(&bars->s_free[1], (ns - 1) & 1))) &&
                        mbar_try_wait(&bars->kv_full[ns % kStages], (ns / kStages) & 1)) {
                        tc_fence_after();
                        const int j = ns;
                        const uint64_t kd = kd0 + (uint64_t)((j % kStages) * (kStageBytes >> 4));
                        // one block's K steps back to back: consecutive MMAs
                        // into one accumulator run at the tensor pipe's rate,
                        // alternating between two accumulators at half of it
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
#pragma unroll
                            for (int k = 0; k < kD / 16; ++k) {
                                const uint64_t koff = (uint64_t)(((k >> 2) * (kKeys * 128) + (k & 3) * 32) >> 4);
                                mma_bf16_ta(tmem + kTmemS + (uint32_t)(u * kKeys),
                                            tmem + kTmemQ + (uint32_t)(u * (kD / 2) + 8 * k), kd + koff,
                                            kIdescS, k > 0 ? 1u : 0u);
                            }
                            mma_commit(&bars->s_full[u]);
                        }
                        ++ns;
                        progressed = true;
                    }
                    if (npv < ns && mbar_try_wait(&bars->p_full[npv & 1], (npv >> 1) & 1) &&
                        mbar_try_wait(&bars->p_full[2 + (npv & 1)], (npv >> 1) & 1)) {
                        tc_fence_after();
                        const int i = npv;
                        const int st = i % kStages;
                        const uint64_t vd = vd0 + (uint64_t)(st * (kStageBytes >> 4));
#pragma unroll
                        for (int k = 0; k < kKeys / 16; ++k) {
#pragma unroll
                            for (int u = 0; u < 2; ++u)
                                mma_bf16(tmem + kTmemO + (uint32_t)(u * kD),
                                         pd0 + (uint64_t)((2 * u + (i & 1)) * (kPBytes >> 4) + k * 2),
                                         vd + (uint64_t)(k * (2048 >> 4)), L::kIdescPV,
                                         (i > 0 || k > 0) ? 1u : 0u);
                        }
                        mma_commit(&bars->p_free[i & 1]);
                        mma_commit(&bars->p_free[2 + (i & 1)]);
                        mma_commit(&bars->kv_empty[st]);
                        ++npv;
                        progressed = true;
                    }
                    if (progressed) {
                        t_last = global_timer_ns();
                    } else if (global_timer_ns() - t_last <= kWaitLimitNs) {
                        // Sleep on the event due first.  Within a tile the
                        // softmax warps release S as soon as they have loaded
                        // it and hand over P only at the end, so while the
                        // next S pair may be issued (at most one ahead of the
                        // PV pairs) its inputs come before the pending P.
                        if (ns < n && ns <= npv + 1) {
                            if (ns > 0 && !mbar_try_wait(&bars->s_free[0], (ns - 1) & 1))
                                (void)mbar_try_wait_sleep(&bars->s_free[0], (ns - 1) & 1, 500u);
                            else if (ns > 0 && !mbar_try_wait(&bars->s_free[1], (ns - 1) & 1))
                                (void)mbar_try_wait_sleep(&bars->s_free[1], (ns - 1) & 1, 500u);
                            else
                                (void)mbar_try_wait_sleep(&bars->kv_full[ns % kStages],
                                                          (ns / kStages) & 1, 200u);
                        } else if (npv < ns) {
                            // a PV pair is next: wait for the block that is not there yet
                            const uint32_t par = (uint32_t)((npv >> 1) & 1);
                            if (mbar_try_wait(&bars->p_full[npv & 1], par))
                                (void)mbar_try_wait_sleep(&bars->p_full[2 + (npv & 1)], par, 500u);
                            else
                                (void)mbar_try_wait_sleep(&bars->p_full[npv & 1], par, 500u);
                        }
                    } else {
                        atomicOr(p.err, kErrWaitTimeout);
                        atomicCAS(p.err + 1, 0u,
                                  0x80000000u | kRoleMma | kBarPFull | (unsigned)(npv & 0xffff));
                        ok = false;
                        break;
                    }
                }
            } else {
                // Issues S_j and PV_i in the order their inputs become ready:
                // S_j needs K/V tile j and its S buffer (group j & 1, buffer
                // (j >> 1) & 1), free once P of tile j - 4 was handed over, i.e.
                // j <= next_pv + 3; PV_i needs P of tile i.
                int next_s = 0, next_pv = 0;
                while (next_pv < n) {
                    bool progressed = false;
                    if (next_s < n && next_s <= next_pv + 3 &&
                        mbar_try_wait(&bars->kv_full[next_s % kStages], (next_s / kStages) & 1)) {
                        tc_fence_after();
                        const int j = next_s;
                        const int sbuf = 2 * (j & 1) + ((j >> 1) & 1);
                        const uint32_t dS = tmem + kTmemS + (uint32_t)(sbuf * kKeys);
                        const uint64_t kd = kd0 + (uint64_t)((j % kStages) * (kStageBytes >> 4));
#pragma unroll
                        for (int k = 0; k < kD / 16; ++k) {
                            const uint64_t qoff = (uint64_t)(((k >> 2) * L::kQBlock + (k & 3) * 32) >> 4);
                            const uint64_t koff = (uint64_t)(((k >> 2) * (kKeys * 128) + (k & 3) * 32) >> 4);
                            mma_bf16(dS, qd0 + qoff, kd + koff, kIdescS, k > 0 ? 1u : 0u);
                        }
                        mma_commit(&bars->s_full[sbuf]);
                        ++next_s;
                        progressed = true;
                    }
                    if (next_pv < next_s &&
                        mbar_try_wait(&bars->p_full[next_pv & 1], (next_pv >> 1) & 1)) {
                        tc_fence_after();
                        const int i = next_pv;
                        const int gr = i & 1;
                        const int st = i % kStages;
                        const uint64_t pd = pd0 + (uint64_t)(gr * (kPBytes >> 4));
                        const uint64_t vd = vd0 + (uint64_t)(st * (kStageBytes >> 4));
                        const uint32_t dO = tmem + kTmemO + (uint32_t)(gr * kD);
#pragma unroll
                        for (int k = 0; k < kKeys / 16; ++k) {
                            mma_bf16(dO, pd + (uint64_t)(k * 2), vd + (uint64_t)(k * (2048 >> 4)),
                                     L::kIdescPV, (i > 1 || k > 0) ? 1u : 0u);
                        }
                        mma_commit(&bars->p_free[gr]);
                        mma_commit(&bars->kv_empty[st]);
                        ++next_pv;
                        progressed = true;
                    }
                    if (progressed) {
                        t_last = global_timer_ns();
                    } else if (global_timer_ns() - t_last <= kWaitLimitNs) {
                        // Nothing ready: suspend on the barrier whose completion
                        // unblocks the most (a pending PV first); the thread
                        // wakes as soon as that phase completes.
                        if (next_pv < next_s)
                            (void)mbar_try_wait_sleep(&bars->p_full[next_pv & 1], (next_pv >> 1) & 1, 500u);
                        else if (next_s < n)
                            (void)mbar_try_wait_sleep(&bars->kv_full[next_s % kStages],
                                                      (next_s / kStages) & 1, 500u);
                    } else {
                        atomicOr(p.err, kErrWaitTimeout);
                        atomicCAS(p.err + 1, 0u,
                                  0x80000000u | kRoleMma | kBarPFull | (unsigned)(next_pv & 0xffff));
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok) bars->abort = 1;
            // drain: every MMA issued so far has completed once this arrives
            mma_commit(&bars->drain);
            mbar_wait_sleep(&bars->drain, 0, p.err, kRoleMma | kBarDrain);
        }
    } else if (warp < kSoftmaxWarps && (warp & 3) < live_quadrants(warp >> 2)) {
        // ------------------------------ softmax warps -------------------------
        // Group gr = warp / 4 takes tiles gr, gr + 2, ... (with ROWS = 256:
        // every tile, for row block gr); warp w owns TMEM lane quadrant w % 4,
        // i.e. rows 32 (w % 4) .. + 31 of the group's 128-row operand.
        const int q4 = warp & 3;
        const int gr = warp >> 2;
        const int r = q4 * 32 + lane;                         // operand row = TMEM lane
        const int rr = (L::kRowGroups ? gr * 128 : 0) + r;    // query row of the CTA
        const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
        const uint32_t o_col = kTmemO + (uint32_t)(gr * kD);
        constexpr bool kPollWaits = L::kActiveQuadrants <= 2 && kD == 128;
        const float c = p.scale_log2;
        const int64_t key_end = ((int64_t)t_end * kKeys < P) ? (int64_t)t_end * kKeys : P;
        // visibility of the n_q speculative keys for this row (the masked tile)
        uint64_t spec_bits = 0;
        if (spec_here && (L::kRowGroups || ((n - 1) & 1) == gr) && rr < Rb) {
            const int iq = (r0 + rr) % p.n_q;
            for (int j = 0; j < p.n_q; ++j) {
                const bool vis =
                    p.mask ? (p.mask[((int64_t)b * p.n_q + iq) * p.n_q + j] != 0) : (j <= iq);
                spec_bits |= (vis ? 1ull : 0ull) << j;
            }
        }
        // A warp whose 32 rows all lie past the CTA's rows computes nothing:
        // it only keeps its place in the barrier protocol.
        const bool idle_warp = rr - lane >= Rb;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        int k_local = 0;
        constexpr int kStep = L::kRowGroups ? 1 : 2;
        for (int i = L::kRowGroups ? 0 : gr; i < n; i += kStep, ++k_local) {
            // 256 rows: one S buffer per block, every phase a tile
            const int sbuf = L::kRowGroups ? gr : 2 * gr + (k_local & 1);
            const uint32_t s_par = L::kRowGroups ? (uint32_t)(k_local & 1) : (uint32_t)((k_local >> 1) & 1);
            const uint32_t s_col = kTmemS + (uint32_t)(sbuf * kKeys);
            ok = __all_sync(0xffffffffu,
                            softmax_wait<kPollWaits>(&bars->s_full[sbuf], s_par, p.err,
                                            kRoleSoftmax | kBarSFull | (unsigned)(i & 0xffff)));
            if (!ok) break;
            if (idle_warp) {
                if constexpr (L::kRowGroups) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->s_free[gr]);
                    // the live warps' order: P buffer k & 1 is handed over
                    // again only after PV_{k-2} has read it
                    if (k_local >= 2) {
                        ok = __all_sync(0xffffffffu,
                                        mbar_wait_sleep(&bars->p_free[2 * gr + (k_local & 1)],
                                                        (uint32_t)(((k_local >> 1) - 1) & 1), p.err,
                                                        kRoleSoftmax | kBarPFree | (unsigned)(i & 0xffff)));
                        if (!ok) break;
                    }
                    mbar_arrive(&bars->p_full[2 * gr + (k_local & 1)]);
                } else {
                    // stay in step with the group's live warps: the next
                    // tile's arrivals must not count for this one
                    mbar_arrive(&bars->p_full[gr]);
                    ok = __all_sync(0xffffffffu,
                                    softmax_wait<kPollWaits>(&bars->p_full[gr], (uint32_t)(k_local & 1), p.err,
                                                    kRoleSoftmax | kBarPFull | (unsigned)(i & 0xffff)));
                    if (!ok) break;
                }
                continue;
            }
            tc_fence_after();
            uint32_t sr[2][32];
            tmem_ld32(lane_addr + s_col, sr[0]);
            tmem_ld32(lane_addr + s_col + 32, sr[1]);
            tmem_wait_ld();
            if constexpr (L::kRowGroups) {
                // S is in registers: the block's next S may overwrite the buffer
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->s_free[gr]);
            }
            uint64_t valid;
            if (i < n_hist) {
                const int64_t nv = key_end - (int64_t)(t_begin + i) * kKeys;
                valid = nv >= 64 ? ~0ull : ((1ull << nv) - 1ull);
            } else {
                valid = spec_bits;
            }
            float sv[64];
            float mt;
            if (valid == ~0ull) {
                // a whole history tile: no mask to apply
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int j = 0; j < 64; j += 4) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) sv[j + u] = __uint_as_float(sr[(j + u) >> 5][(j + u) & 31]);
                    mx0 = fmax3(mx0, sv[j], sv[j + 1]);
                    mx1 = fmax3(mx1, sv[j + 2], sv[j + 3]);
                }
                mt = fmaxf(mx0, mx1) * c;
            } else {
                float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
                for (int j = 0; j < 64; j += 4) {
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        sv[j + u] = ((valid >> (j + u)) & 1ull)
                                        ? __uint_as_float(sr[(j + u) >> 5][(j + u) & 31])
                                        : -INFINITY;
                    mx0 = fmaxf(mx0, sv[j]);
                    mx1 = fmaxf(mx1, sv[j + 1]);
                    mx2 = fmaxf(mx2, sv[j + 2]);
                    mx3 = fmaxf(mx3, sv[j + 3]);
                }
                mt = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c;
            }
            float corr = 1.f;
            bool rescale = false;
            if (mt > m_run + 8.f) {               // also true for the first finite tile
                corr = ex2(m_run - mt);           // 0 when m_run = -inf
                rescale = (k_local > 0);
                m_run = mt;
            }
            // a row that has seen no visible key yet (a speculative tile whose
            // mask hides every key from it, with no history before it) keeps
            // p = 0 instead of exp(-inf + inf)
            const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
            // packed f32x2 arithmetic: the same per-lane fma and adds, half the instructions
            const float2 c2 = make_float2(c, c), nm2 = make_float2(neg_m, neg_m);
            float2 s01 = make_float2(0.f, 0.f), s23 = make_float2(0.f, 0.f);
            uint32_t pk[32];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float2 x01 = fma2(make_float2(sv[2 * j], sv[2 * j + 1]), c2, nm2);
                const float2 x23 = fma2(make_float2(sv[2 * j + 2], sv[2 * j + 3]), c2, nm2);
                const float2 p01 = make_float2(ex2(x01.x), ex2(x01.y));
                const float2 p23 = make_float2(ex2(x23.x), ex2(x23.y));
                s01 = add2(s01, p01);
                s23 = add2(s23, p23);
                pk[j] = pack_bf16x2(p01.x, p01.y);
                pk[j + 1] = pack_bf16x2(p23.x, p23.y);
            }
            l_run = l_run * corr + ((s01.x + s01.y) + (s23.x + s23.y));
            const bool any_rescale = __any_sync(0xffffffffu, rescale);
            if constexpr (L::kRowGroups) {
                // P buffer k & 1 was last read by PV_{k-2}; rescaling O also
                // needs PV_{k-1} to have accumulated into it
                if (k_local >= 2) {
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait_sleep(&bars->p_free[2 * gr + (k_local & 1)],
                                                    (uint32_t)(((k_local >> 1) - 1) & 1), p.err,
                                                    kRoleSoftmax | kBarPFree | (unsigned)(i & 0xffff)));
                    if (!ok) break;
                }
                if (any_rescale) {
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait_sleep(&bars->p_free[2 * gr + ((k_local - 1) & 1)],
                                                    (uint32_t)(((k_local - 1) >> 1) & 1), p.err,
                                                    kRoleSoftmax | kBarPFree | (unsigned)(i & 0xffff)));
                    if (!ok) break;
                }
                tc_fence_after();
            } else if (k_local > 0) {
                // the previous PV of this group read P and accumulated into O
                ok = __all_sync(0xffffffffu,
                                softmax_wait<kPollWaits>(&bars->p_free[gr], (k_local - 1) & 1, p.err,
                                                kRoleSoftmax | kBarPFree | (unsigned)(i & 0xffff)));
                if (!ok) break;
                tc_fence_after();
            }
            if (any_rescale) {
#pragma unroll
                for (int qq = 0; qq < kD / 32; ++qq) {
                    uint32_t o[32];
                    tmem_ld32(lane_addr + o_col + qq * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * corr);
                    tmem_st32(lane_addr + o_col + qq * 32, o);
                }
                tmem_wait_st();
            }
            const int pbuf = L::kRowGroups ? 2 * gr + (k_local & 1) : gr;
            uint8_t* prow = smem + kOffP + pbuf * kPBytes + r * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                *reinterpret_cast<uint4*>(prow + ((j ^ (r & 7)) << 4)) =
                    make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bars->p_full[L::kRowGroups ? 2 * gr + (k_local & 1) : gr]);
        }
        if (tid == 0) griddep_launch_dependents();
        // Wait for this group's last PV, publish (m, l), then combine both
        // groups' O columns: warp w writes columns 64 (w / 4) .. + 63 of its rows.
        if (ok && k_local > 0) {
            // 256 rows: the block's last PV read P buffer (k - 1) & 1
            const int fb = L::kRowGroups ? 2 * gr + ((k_local - 1) & 1) : gr;
            const uint32_t fpar = L::kRowGroups ? (uint32_t)(((k_local - 1) >> 1) & 1)
                                                : (uint32_t)((k_local - 1) & 1);
            ok = __all_sync(0xffffffffu, softmax_wait<kPollWaits>(&bars->p_free[fb], fpar, p.err,
                                                         kRoleSoftmax | kBarPFree | 0xffffu));
        }
        if constexpr (L::kRowGroups) {
            // Each group owns its rows' partial: (O, m, l) as they stand.
            if (ok) {
                tc_fence_after();
                const bool real_row = rr < Rb;
                const bool has = k_local > 0 && l_run > 0.f;
                float* dst = p.part_acc + (slot + r0 + rr) * kD;
#pragma unroll
                for (int qq = 0; qq < kD / 32; ++qq) {
                    uint32_t o[32];
                    tmem_ld32(lane_addr + o_col + qq * 32, o);
                    tmem_wait_ld();
                    if (real_row) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4) {
                            float4 v;
                            v.x = has ? __uint_as_float(o[j]) : 0.f;
                            v.y = has ? __uint_as_float(o[j + 1]) : 0.f;
                            v.z = has ? __uint_as_float(o[j + 2]) : 0.f;
                            v.w = has ? __uint_as_float(o[j + 3]) : 0.f;
                            *reinterpret_cast<float4*>(dst + qq * 32 + j) = v;
                        }
                    }
                }
                if (real_row) {
                    p.part_ml[(slot + r0 + rr) * 2 + 0] = k_local > 0 ? m_run : -INFINITY;
                    p.part_ml[(slot + r0 + rr) * 2 + 1] = k_local > 0 ? l_run : 0.f;
                }
            }
            if (!ok) bars->abort = 1;
        } else {
        // (m, l) of this group go into its own P buffer, which its last PV
        // product has finished reading.
        float* pub = reinterpret_cast<float*>(smem + kOffP + gr * kPBytes);
        if (ok) {
            pub[r] = k_local > 0 ? m_run : -INFINITY;
            pub[128 + r] = k_local > 0 ? l_run : 0.f;
        }
        if (!ok && lane == 0) bars->grp_ok[gr] = 0;   // any warp of the group can veto
        asm volatile("bar.sync 1, %0;" ::"r"(2 * 32 * live_quadrants(0)) : "memory");
        ok = bars->grp_ok[0] && bars->grp_ok[1];
        if (ok) {
            tc_fence_after();
            const float* pub0 = reinterpret_cast<const float*>(smem + kOffP);
            const float* pub1 = reinterpret_cast<const float*>(smem + kOffP + kPBytes);
            const float m0 = pub0[r], m1 = pub1[r];
            const float l0 = pub0[128 + r], l1 = pub1[128 + r];
            const float M = fmaxf(m0, m1);
            const bool has0 = l0 > 0.f, has1 = l1 > 0.f;
            const float w0 = has0 ? ex2(m0 - M) : 0.f;
            const float w1 = has1 ? ex2(m1 - M) : 0.f;
            // tcgen05.ld is warp-collective (.sync.aligned): every lane
            // executes the same loads; only the stores are per-row.
            const bool real_row = r < Rb;
            const int half = gr;                      // this warp's D / 2 output columns
            const int c0 = half * (kD / 2);
            float* dst = p.part_acc + (slot + r0 + r) * kD + c0;
#pragma unroll
            for (int qq = 0; qq < kD / 64; ++qq) {
                uint32_t o0[32], o1[32];
                tmem_ld32(lane_addr + kTmemO + c0 + qq * 32, o0);
                tmem_ld32(lane_addr + kTmemO + kD + c0 + qq * 32, o1);
                tmem_wait_ld();
                if (real_row) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        float4 v;
                        v.x = (has0 ? w0 * __uint_as_float(o0[j]) : 0.f) + (has1 ? w1 * __uint_as_float(o1[j]) : 0.f);
                        v.y = (has0 ? w0 * __uint_as_float(o0[j + 1]) : 0.f) + (has1 ? w1 * __uint_as_float(o1[j + 1]) : 0.f);
                        v.z = (has0 ? w0 * __uint_as_float(o0[j + 2]) : 0.f) + (has1 ? w1 * __uint_as_float(o1[j + 2]) : 0.f);
                        v.w = (has0 ? w0 * __uint_as_float(o0[j + 3]) : 0.f) + (has1 ? w1 * __uint_as_float(o1[j + 3]) : 0.f);
                        *reinterpret_cast<float4*>(dst + qq * 32 + j) = v;
                    }
                }
            }
            if (real_row && half == 0) {
                p.part_ml[(slot + r0 + r) * 2 + 0] = M;
                p.part_ml[(slot + r0 + r) * 2 + 1] = l0 * w0 + l1 * w1;
            }
        }
        if (!ok) bars->abort = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// 2-D view [rows, d] of a bf16 KV cache; 64 x 64 boxes, 128-byte swizzle.
bool make_kv_map(CUtensorMap* m, const void* base, uint64_t rows, int d) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kKeys};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool attn_prefix_tc_supported(const AttnParams& p, int dtype) {
    if (dtype != 1 || (p.d != 64 && p.d != 128)) return false;
    if (p.R < 1 || p.R > 512) return false;      // up to two 256-row blocks
    if ((int64_t)p.B * p.Hkv * p.cap >= ((int64_t)1 << 31)) return false;
    return tensor_map_encoder() != nullptr;
}

namespace {

template <int ROWS, int D>
cudaError_t launch_rows(const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnParams& p,
                        cudaStream_t st) {
    auto kern = attn_prefix_tc_kernel<ROWS, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Plan<ROWS, D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.S * tc_row_blocks(p.R), p.Hkv, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Plan<ROWS, D>::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmK, tmV, p);
}

}  // namespace

cudaError_t launch_attn_prefix_tc(const AttnParams& p, cudaStream_t st) {
    CUtensorMap tmK, tmV;
    const uint64_t rows = (uint64_t)p.B * p.Hkv * p.cap;
    if (!make_kv_map(&tmK, p.K, rows, p.d) || !make_kv_map(&tmV, p.V, rows, p.d))
        return cudaErrorInvalidValue;
    if (p.d == 64) {
        if (p.R <= 64) return launch_rows<64, 64>(tmK, tmV, p, st);
        return p.R <= 128 ? launch_rows<128, 64>(tmK, tmV, p, st) : launch_rows<256, 64>(tmK, tmV, p, st);
    }
    if (p.R <= 64) return launch_rows<64, 128>(tmK, tmV, p, st);
    return p.R <= 128 ? launch_rows<128, 128>(tmK, tmV, p, st) : launch_rows<256, 128>(tmK, tmV, p, st);
}

}  // namespace rapid
