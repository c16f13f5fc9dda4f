// C ABI of librapid.so: argument checks, workspace planning, launches.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "accept.cuh"
#include "attn.cuh"
#include "common.cuh"
#include "kv_commit.cuh"
#include "lm_head.cuh"
#include "lse_merge.cuh"
#include "retrieval.cuh"
#include "rapid.h"

namespace rapid {

// [0] sticky error bits, [1] code of the first timed-out wait, [2..7] spare.
__device__ unsigned int g_device_error[8] = {0, 0, 0, 0, 0, 0, 0, 0};

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

unsigned int* device_error_word() {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_error) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return static_cast<unsigned int*>(ptr);
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 148;
    return n;
}

struct AttnPlan {
    bool tc;        // tensor-core history kernel
    int S;          // splits of the history per (b, kv head)
    int nparts;     // partial slots per (b, kv head); per kv head for the tensor-core kernel
    int64_t chunk;  // history rows per split
    size_t part_rows;   // partial rows in the workspace
    size_t ws_bytes;
};

bool attn_args_ok(int B, int Hq, int Hkv, int d, int n_q, int64_t cap, int dtype) {
    if (B < 1 || Hq < 1 || Hkv < 1 || (Hq % Hkv) != 0) return false;
    if ((int64_t)B * Hkv > 65535) return false;   // one grid dimension of the merge launch
    if (d != 64 && d != 128) return false;
    if (n_q < 1 || n_q > RAPID_MAX_NQ) return false;
    if (cap < n_q || cap > ((int64_t)1 << 31)) return false;
    if (dtype != RAPID_DTYPE_F32 && dtype != RAPID_DTYPE_BF16) return false;
    const int64_t R = (int64_t)(Hq / Hkv) * n_q;
    if (R > 4096) return false;
    return true;
}

AttnPlan plan_attn(int B, int Hq, int Hkv, int d, int n_q, int64_t cap, int dtype) {
    AttnPlan pl{};
    const int G = Hq / Hkv;
    const int R = G * n_q;
    AttnParams probe{};
    probe.B = B; probe.Hq = Hq; probe.Hkv = Hkv; probe.d = d; probe.n_q = n_q; probe.G = G;
    probe.R = R; probe.cap = cap;
    pl.tc = attn_prefix_tc_supported(probe, dtype);
    const int64_t max_prefix = cap - n_q;
    const int sms = sm_count();
    int64_t chunk;
    if (pl.tc) {
        // One CTA per SM, one wave: (sequence, split) slots per KV head, times
        // the row blocks of a wide group.  The kernel decides on the device
        // how the slots are shared out over the sequences.
        const int64_t per_slot = (int64_t)Hkv * tc_row_blocks(R);
        int64_t S = sms / per_slot;
        if (S < B) S = B;
        pl.S = (int)S;
        pl.nparts = (int)S;
        pl.chunk = 0;
        // partials by launch slot: [Hkv, S, R] rows, whatever B is
        const size_t part = (size_t)Hkv * pl.nparts * R;
        pl.part_rows = part;
        pl.ws_bytes = align_up(part * d * sizeof(float)) + align_up(part * 2 * sizeof(float)) +
                      2 * align_up((size_t)B * Hkv * sizeof(int));
        return pl;
    } else {
        const int64_t rbs = (R + 63) / 64;
        const int64_t ctas = (int64_t)B * Hkv * rbs;
        int64_t S = (4 * (int64_t)sms + ctas - 1) / ctas;
        if (S < 1) S = 1;
        chunk = (max_prefix + S - 1) / S;
    }
    chunk = (chunk + 127) / 128 * 128;
    if (chunk < 128) chunk = 128;
    int64_t S = (max_prefix + chunk - 1) / chunk;
    if (S < 1) S = 1;
    if (S > 512) {   // the merge kernel stages at most 1024 partial weights per row
        S = 512;
        chunk = ((max_prefix + S - 1) / S + 127) / 128 * 128;
        S = (max_prefix + chunk - 1) / chunk;
    }
    pl.S = (int)S;
    pl.chunk = chunk;
    pl.nparts = (int)S;
    const size_t part = (size_t)B * Hkv * pl.nparts * R;
    pl.part_rows = part;
    pl.ws_bytes = align_up(part * d * sizeof(float)) + align_up(part * 2 * sizeof(float)) +
                  2 * align_up((size_t)B * Hkv * sizeof(int));
    return pl;
}

// The acceptance launch after argument checks (shared by rapid_accept and
// rapid_lm_head_accept).
rapid_status accept_launch(const float* z_target, const float* q_draft,
                           const int32_t* draft_tokens, const int32_t* parent, int B, int n_q,
                           const int32_t* n_nodes, int V, float T, float eta,
                           uint64_t philox_seed, const uint64_t* philox_seed_dev, uint32_t flags,
                           int32_t* n_accepted, int32_t* next_token, int32_t* path, float* diag,
                           void* workspace, cudaStream_t st) {
    AcceptShape sh{};
    if (accept_plan(V, B * n_q, &sh) != cudaSuccess) {
        (void)cudaGetLastError();
        return RAPID_EUNSUPPORTED;
    }
    const size_t rows = (size_t)B * n_q;
    char* ws = static_cast<char*>(workspace);
    AcceptParams p{};
    p.z = z_target; p.q = q_draft; p.tokens = draft_tokens; p.parent = parent;
    p.ws_accept = reinterpret_cast<int32_t*>(ws);
    ws += align_up(rows * sizeof(int32_t));
    p.ws_stats = reinterpret_cast<float*>(ws);
    p.diag = diag; p.n_accepted = n_accepted; p.next_token = next_token; p.path = path;
    p.B = B; p.n_q = n_q; p.V = V;
    p.bulk = ((V % 4) == 0 && aligned16(z_target) && aligned16(q_draft)) ? 1 : 0;
    p.clamp = (flags & RAPID_ACCEPT_TAIL_CLAMP) ? 1 : 0;
    p.invT = 1.0f / T;
    p.eta = eta;
    p.seed_lo = (uint32_t)(philox_seed & 0xffffffffu);
    p.seed_hi = (uint32_t)(philox_seed >> 32);
    p.seed_dev = reinterpret_cast<const unsigned long long*>(philox_seed_dev);
    p.n_nodes = n_nodes;
    p.err = device_error_word();
    return launch_accept(p, sh, st) == cudaSuccess ? RAPID_OK : RAPID_ECUDA;
}

// Self-test of the bounded waits (rapid_wait_selftest): a copy in flight,
// then a wait on a phase nothing completes, which must give up, record its
// code and let the copy land before the CTA leaves.
constexpr unsigned int kSelftestCode = 0x47000001u;   // recorded as 0xC7000001
__device__ __align__(16) unsigned char g_selftest_src[1024];

__global__ void wait_selftest_kernel(unsigned int* err, uint64_t limit_ns) {
    __shared__ __align__(128) unsigned char buf[1024];
    __shared__ __align__(8) uint64_t copied;
    __shared__ __align__(8) uint64_t never;
    if (threadIdx.x == 0) {
        mbar_init(&copied, 1);
        mbar_init(&never, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&copied, (uint32_t)sizeof(buf));
        bulk_g2s(buf, g_selftest_src, (uint32_t)sizeof(buf), &copied);
        (void)mbar_wait(&never, 0u, err, kSelftestCode, limit_ns);
        (void)mbar_wait(&copied, 0u, err, kSelftestCode + 1u);
    }
    __syncthreads();
}

bool lm_head_args_ok(int rows, int hidden_dim, int V) {
    if (rows < 1 || rows > RAPID_LM_HEAD_MAX_ROWS) return false;
    if (hidden_dim < 64 || hidden_dim > RAPID_LM_HEAD_MAX_HIDDEN || hidden_dim % 64 != 0) return false;
    if (V < 1 || V > RAPID_LM_HEAD_MAX_VOCAB) return false;
    return true;
}

}  // namespace
}  // namespace rapid

using namespace rapid;

extern "C" {

size_t rapid_verify_attn_workspace_size(int B, int Hq, int Hkv, int d, int n_q,
                                        int64_t kv_capacity, int dtype) {
    if (!attn_args_ok(B, Hq, Hkv, d, n_q, kv_capacity, dtype)) return 0;
    return plan_attn(B, Hq, Hkv, d, n_q, kv_capacity, dtype).ws_bytes;
}

rapid_status rapid_verify_attn(const void* Q, const void* Kcache, const void* Vcache, int dtype,
                               int B, int Hq, int Hkv, int d, int n_q, int64_t kv_capacity,
                               const int32_t* prefix_len, const uint8_t* spec_mask,
                               float softmax_scale, void* O, float* LSE, void* workspace,
                               size_t workspace_bytes, void* stream) {
    if (!Q || !Kcache || !Vcache || !prefix_len || !O || !LSE || !workspace) return RAPID_EINVAL;
    if (!attn_args_ok(B, Hq, Hkv, d, n_q, kv_capacity, dtype)) return RAPID_EINVAL;
    if (!aligned16(Q) || !aligned16(Kcache) || !aligned16(Vcache) || !aligned16(O) ||
        !aligned16(workspace) || (reinterpret_cast<uintptr_t>(LSE) & 3u))
        return RAPID_EINVAL;
    if (!std::isfinite(softmax_scale)) return RAPID_EINVAL;
    const AttnPlan pl = plan_attn(B, Hq, Hkv, d, n_q, kv_capacity, dtype);
    if (workspace_bytes < pl.ws_bytes) return RAPID_ENOMEM;

    AttnParams p{};
    p.Q = Q; p.K = Kcache; p.V = Vcache; p.prefix_len = prefix_len; p.mask = spec_mask;
    p.O = O; p.LSE = LSE;
    p.cap = kv_capacity; p.chunk = pl.chunk;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.d = d; p.n_q = n_q; p.G = Hq / Hkv; p.R = p.G * n_q;
    p.S = pl.S;
    p.spec_in_partials = pl.tc ? 1 : 0;
    p.balanced = pl.tc ? 1 : 0;
    p.nparts = pl.nparts;
    p.err = device_error_word();
    p.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt((float)d);
    p.scale_log2 = p.scale * kLog2e;
    const size_t part = pl.part_rows;
    char* ws = static_cast<char*>(workspace);
    p.part_acc = reinterpret_cast<float*>(ws);
    ws += align_up(part * d * sizeof(float));
    p.part_ml = reinterpret_cast<float*>(ws);
    ws += align_up(part * 2 * sizeof(float));
    p.part_nsplit = reinterpret_cast<int*>(ws);
    ws += align_up((size_t)B * Hkv * sizeof(int));
    p.part_first = reinterpret_cast<int*>(ws);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = pl.tc ? launch_attn_prefix_tc(p, st) : launch_attn_prefix_simt(p, dtype, st);
    if (e != cudaSuccess) return RAPID_ECUDA;
    e = launch_attn_merge(p, dtype, st);
    return e == cudaSuccess ? RAPID_OK : RAPID_ECUDA;
}

rapid_status rapid_attn_merge(const void* O_parts, const float* LSE_parts, int dtype,
                              int n_parts, int64_t rows, int d, void* O, float* LSE,
                              void* stream) {
    if (!O_parts || !LSE_parts || !O || !LSE) return RAPID_EINVAL;
    if (dtype != RAPID_DTYPE_F32 && dtype != RAPID_DTYPE_BF16) return RAPID_EINVAL;
    if (n_parts < 1 || rows < 1 || (d != 64 && d != 128)) return RAPID_EINVAL;
    if (rows > (int64_t)1 << 36) return RAPID_EINVAL;
    if (!aligned16(O_parts) || !aligned16(O) || (reinterpret_cast<uintptr_t>(LSE_parts) & 3u) ||
        (reinterpret_cast<uintptr_t>(LSE) & 3u))
        return RAPID_EINVAL;
    return launch_lse_merge(O_parts, LSE_parts, dtype == RAPID_DTYPE_BF16, n_parts, rows, d, O, LSE,
                            static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? RAPID_OK
               : RAPID_ECUDA;
}

size_t rapid_accept_workspace_size(int B, int n_q, int V) {
    if (B < 1 || n_q < 1 || n_q > RAPID_MAX_NQ || V < 1 || V > RAPID_MAX_VOCAB) return 0;
    const size_t rows = (size_t)B * n_q;
    return align_up(rows * sizeof(int32_t)) + align_up(rows * 4 * sizeof(float));
}

// Host checks shared by rapid_accept and rapid_accept_ex.
static rapid_status accept_args(const float* z_target, const float* q_draft,
                                const int32_t* draft_tokens, int B, int n_q, int V, float T,
                                float eta, uint32_t flags, const int32_t* n_accepted,
                                const int32_t* next_token, const void* workspace,
                                size_t workspace_bytes) {
    if (!z_target || !q_draft || !draft_tokens || !n_accepted || !next_token || !workspace)
        return RAPID_EINVAL;
    if (B < 1 || n_q < 1 || n_q > RAPID_MAX_NQ || V < 1 || V > RAPID_MAX_VOCAB) return RAPID_EINVAL;
    if (B > 65535) return RAPID_EINVAL;   // one grid dimension of the selection launch
    if (!(T > 0.f) || !std::isfinite(T) || !(eta >= 0.f) || !std::isfinite(eta)) return RAPID_EINVAL;
    if ((flags & ~(uint32_t)RAPID_ACCEPT_TAIL_CLAMP) != 0) return RAPID_EINVAL;
    if ((reinterpret_cast<uintptr_t>(z_target) & 3u) || (reinterpret_cast<uintptr_t>(q_draft) & 3u))
        return RAPID_EINVAL;
    const size_t need = rapid_accept_workspace_size(B, n_q, V);
    if (workspace_bytes < need) return RAPID_ENOMEM;
    if (reinterpret_cast<uintptr_t>(workspace) & 15u) return RAPID_EINVAL;
    return RAPID_OK;
}

rapid_status rapid_accept(const float* z_target, const float* q_draft, const int32_t* draft_tokens,
                          const int32_t* parent, int B, int n_q, int V, float T, float eta,
                          uint64_t philox_seed, uint32_t flags, int32_t* n_accepted,
                          int32_t* next_token, int32_t* path, float* diag, void* workspace,
                          size_t workspace_bytes, void* stream) {
    const rapid_status s = accept_args(z_target, q_draft, draft_tokens, B, n_q, V, T, eta, flags,
                                       n_accepted, next_token, workspace, workspace_bytes);
    if (s != RAPID_OK) return s;
    return accept_launch(z_target, q_draft, draft_tokens, parent, B, n_q, nullptr, V, T, eta,
                         philox_seed, nullptr, flags, n_accepted, next_token, path, diag,
                         workspace, static_cast<cudaStream_t>(stream));
}

rapid_status rapid_accept_ex(const float* z_target, const float* q_draft,
                             const int32_t* draft_tokens, const int32_t* parent,
                             const int32_t* n_nodes, int B, int n_q, int V, float T, float eta,
                             uint64_t philox_seed, const uint64_t* philox_seed_dev,
                             uint32_t flags, int32_t* n_accepted, int32_t* next_token,
                             int32_t* path, float* diag, void* workspace,
                             size_t workspace_bytes, void* stream) {
    if (philox_seed_dev && (reinterpret_cast<uintptr_t>(philox_seed_dev) & 7u))
        return RAPID_EINVAL;
    if (n_nodes && (reinterpret_cast<uintptr_t>(n_nodes) & 3u)) return RAPID_EINVAL;
    const rapid_status s = accept_args(z_target, q_draft, draft_tokens, B, n_q, V, T, eta, flags,
                                       n_accepted, next_token, workspace, workspace_bytes);
    if (s != RAPID_OK) return s;
    return accept_launch(z_target, q_draft, draft_tokens, parent, B, n_q, n_nodes, V, T, eta,
                         philox_seed, philox_seed_dev, flags, n_accepted, next_token, path, diag,
                         workspace, static_cast<cudaStream_t>(stream));
}

rapid_status rapid_lm_head(const void* hidden, const void* W_lm, int rows, int hidden_dim, int V,
                           float* z, void* stream) {
    if (!hidden || !W_lm || !z) return RAPID_EINVAL;
    if (!lm_head_args_ok(rows, hidden_dim, V)) return RAPID_EINVAL;
    if (!aligned16(hidden) || !aligned16(W_lm) || (reinterpret_cast<uintptr_t>(z) & 3u))
        return RAPID_EINVAL;
    if (!lm_head_supported()) return RAPID_EUNSUPPORTED;
    return launch_lm_head(hidden, W_lm, rows, hidden_dim, V, z, device_error_word(),
                          static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? RAPID_OK
               : RAPID_ECUDA;
}

size_t rapid_lm_head_accept_workspace_size(int B, int n_q, int V) {
    const size_t acc = rapid_accept_workspace_size(B, n_q, V);
    if (acc == 0 || (int64_t)B * n_q > RAPID_LM_HEAD_MAX_ROWS) return 0;
    return align_up((size_t)B * n_q * V * sizeof(float)) + acc;
}

static rapid_status lm_head_accept_impl(const void* hidden, const void* W_lm, int hidden_dim,
                                        const float* q_draft, const int32_t* draft_tokens,
                                        const int32_t* parent, const int32_t* n_nodes, int B,
                                        int n_q, int V, float T, float eta, uint64_t philox_seed,
                                        const uint64_t* philox_seed_dev, uint32_t flags,
                                        int32_t* n_accepted, int32_t* next_token, int32_t* path,
                                        float* diag, void* workspace, size_t workspace_bytes,
                                        void* stream) {
    if (!hidden || !W_lm || !q_draft || !draft_tokens || !n_accepted || !next_token || !workspace)
        return RAPID_EINVAL;
    if (B < 1 || n_q < 1 || n_q > RAPID_MAX_NQ || V < 1 || V > RAPID_MAX_VOCAB) return RAPID_EINVAL;
    if ((int64_t)B * n_q > RAPID_LM_HEAD_MAX_ROWS || !lm_head_args_ok(B * n_q, hidden_dim, V))
        return RAPID_EINVAL;
    if (!(T > 0.f) || !std::isfinite(T) || !(eta >= 0.f) || !std::isfinite(eta)) return RAPID_EINVAL;
    if ((flags & ~(uint32_t)RAPID_ACCEPT_TAIL_CLAMP) != 0) return RAPID_EINVAL;
    if (!aligned16(hidden) || !aligned16(W_lm) || (reinterpret_cast<uintptr_t>(q_draft) & 3u) ||
        !aligned16(workspace))
        return RAPID_EINVAL;
    if (philox_seed_dev && (reinterpret_cast<uintptr_t>(philox_seed_dev) & 7u)) return RAPID_EINVAL;
    if (n_nodes && (reinterpret_cast<uintptr_t>(n_nodes) & 3u)) return RAPID_EINVAL;
    if (workspace_bytes < rapid_lm_head_accept_workspace_size(B, n_q, V)) return RAPID_ENOMEM;
    if (!lm_head_supported()) return RAPID_EUNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Up to 16 rows: one cooperative kernel does the product and the
    // acceptance step, z stays in shared memory (its scratch is a prefix of
    // the workspace that the two-launch form below uses for z).
    {
        LmAcceptParams fa{};
        fa.q = q_draft; fa.tokens = draft_tokens; fa.parent = parent; fa.n_nodes = n_nodes;
        fa.seed_dev = reinterpret_cast<const unsigned long long*>(philox_seed_dev);
        fa.n_accepted = n_accepted; fa.next_token = next_token; fa.path = path; fa.diag = diag;
        fa.B = B; fa.n_q = n_q;
        fa.clamp = (flags & RAPID_ACCEPT_TAIL_CLAMP) ? 1 : 0;
        fa.invT = 1.0f / T;
        fa.eta = eta;
        fa.seed_lo = (uint32_t)(philox_seed & 0xffffffffu);
        fa.seed_hi = (uint32_t)(philox_seed >> 32);
        const cudaError_t e = launch_lm_head_accept(hidden, W_lm, hidden_dim, V, fa, workspace,
                                                    workspace_bytes, device_error_word(), st);
        if (e == cudaSuccess) return RAPID_OK;
        if (e != cudaErrorNotSupported) return RAPID_ECUDA;
    }
    // z lives at the front of the workspace (B n_q V floats, L2-resident at
    // the sizes of one verify step); the acceptance scratch follows it.
    float* z = static_cast<float*>(workspace);
    void* acc_ws = static_cast<char*>(workspace) + align_up((size_t)B * n_q * V * sizeof(float));
    if (launch_lm_head(hidden, W_lm, B * n_q, hidden_dim, V, z, device_error_word(), st) !=
        cudaSuccess)
        return RAPID_ECUDA;
    return accept_launch(z, q_draft, draft_tokens, parent, B, n_q, n_nodes, V, T, eta,
                         philox_seed, philox_seed_dev, flags, n_accepted, next_token, path, diag,
                         acc_ws, st);
}

rapid_status rapid_lm_head_accept(const void* hidden, const void* W_lm, int hidden_dim,
                                  const float* q_draft, const int32_t* draft_tokens,
                                  const int32_t* parent, int B, int n_q, int V, float T, float eta,
                                  uint64_t philox_seed, uint32_t flags, int32_t* n_accepted,
                                  int32_t* next_token, int32_t* path, float* diag,
                                  void* workspace, size_t workspace_bytes, void* stream) {
    return lm_head_accept_impl(hidden, W_lm, hidden_dim, q_draft, draft_tokens, parent, nullptr,
                               B, n_q, V, T, eta, philox_seed, nullptr, flags, n_accepted,
                               next_token, path, diag, workspace, workspace_bytes, stream);
}

rapid_status rapid_lm_head_accept_ex(const void* hidden, const void* W_lm, int hidden_dim,
                                     const float* q_draft, const int32_t* draft_tokens,
                                     const int32_t* parent, const int32_t* n_nodes, int B,
                                     int n_q, int V, float T, float eta, uint64_t philox_seed,
                                     const uint64_t* philox_seed_dev, uint32_t flags,
                                     int32_t* n_accepted, int32_t* next_token, int32_t* path,
                                     float* diag, void* workspace, size_t workspace_bytes,
                                     void* stream) {
    return lm_head_accept_impl(hidden, W_lm, hidden_dim, q_draft, draft_tokens, parent, n_nodes,
                               B, n_q, V, T, eta, philox_seed, philox_seed_dev, flags,
                               n_accepted, next_token, path, diag, workspace, workspace_bytes,
                               stream);
}

const char* rapid_status_string(int status) {
    switch (status) {
        case RAPID_OK: return "ok";
        case RAPID_EINVAL: return "invalid argument";
        case RAPID_ECUDA: return "CUDA error";
        case RAPID_ENOMEM: return "workspace too small";
        case RAPID_ETIMEOUT: return "a bounded wait inside a kernel gave up";
        case RAPID_EUNSUPPORTED: return "unsupported shape";
        default: return "unknown status";
    }
}

int rapid_version(void) { return 200; }

rapid_status rapid_kv_commit(void* const* K_layers, void* const* V_layers, int layers, int dtype,
                             int B, int Hkv, int d, int64_t kv_capacity, int n_q,
                             const int32_t* prefix_len, const int32_t* path,
                             const int32_t* n_accepted, void* stream) {
    if (!K_layers || !V_layers || !prefix_len || !path || !n_accepted) return RAPID_EINVAL;
    if (layers < 1 || layers > RAPID_COMMIT_MAX_LAYERS || B < 1 || Hkv < 1) return RAPID_EINVAL;
    if ((d != 64 && d != 128) || n_q < 1 || n_q > RAPID_MAX_NQ || kv_capacity < 1) return RAPID_EINVAL;
    if (dtype != RAPID_DTYPE_F32 && dtype != RAPID_DTYPE_BF16) return RAPID_EINVAL;
    CommitParams p{};
    for (int l = 0; l < layers; ++l) {
        if (!K_layers[l] || !V_layers[l] || !aligned16(K_layers[l]) || !aligned16(V_layers[l]))
            return RAPID_EINVAL;
        p.K[l] = K_layers[l];
        p.V[l] = V_layers[l];
    }
    if (n_q == 1) return RAPID_OK;   // no draft node: nothing can move
    p.prefix_len = prefix_len;
    p.path = path;
    p.n_acc = n_accepted;
    p.err = device_error_word();
    p.cap = kv_capacity;
    p.layers = layers;
    p.B = B;
    p.Hkv = Hkv;
    p.n_q = n_q;
    p.row_bytes = d * (dtype == RAPID_DTYPE_BF16 ? 2 : 4);
    return launch_kv_commit(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? RAPID_OK
                                                                                 : RAPID_ECUDA;
}

rapid_status rapid_kv_advance(int32_t* prefix_len, const int32_t* n_accepted, int B, int n_q,
                              int64_t kv_capacity, void* stream) {
    if (!prefix_len || !n_accepted || B < 1 || n_q < 1 || n_q > RAPID_MAX_NQ || kv_capacity < 1)
        return RAPID_EINVAL;
    return launch_kv_advance(prefix_len, n_accepted, B, n_q, kv_capacity, device_error_word(),
                             static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? RAPID_OK
               : RAPID_ECUDA;
}

rapid_status rapid_retrieval_scores(const void* query, const void* chunks, int dtype, int B, int N,
                                    int D, float* scores, void* stream) {
    if (!query || !chunks || !scores || B < 1 || N < 1) return RAPID_EINVAL;
    if (D < 8 || D > 8192 || D % 8 != 0) return RAPID_EINVAL;
    if (dtype != RAPID_DTYPE_F32 && dtype != RAPID_DTYPE_BF16) return RAPID_EINVAL;
    if (!aligned16(query) || !aligned16(chunks)) return RAPID_EINVAL;
    return launch_retrieval_scores(query, chunks, dtype, B, N, D, scores,
                                   static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? RAPID_OK
               : RAPID_ECUDA;
}

rapid_status rapid_retrieval_select(const float* scores, const int32_t* context_tokens, int B, int N,
                                    int chunk_tokens, float threshold, int min_tokens, int ratio,
                                    int32_t* selected, int32_t* n_selected,
                                    int32_t* tokens_selected, void* stream) {
    if (!scores || !context_tokens || !selected || !n_selected || !tokens_selected) return RAPID_EINVAL;
    if (B < 1 || N < 1 || N > RAPID_RETRIEVAL_MAX_CHUNKS || chunk_tokens < 1 || ratio < 1 ||
        min_tokens < 0)
        return RAPID_EINVAL;
    return launch_retrieval_select(scores, context_tokens, B, N, chunk_tokens, threshold, min_tokens,
                                   ratio, selected, n_selected, tokens_selected, device_error_word(),
                                   static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? RAPID_OK
               : RAPID_ECUDA;
}


int rapid_device_error(int clear) {
    uint32_t w[8];
    if (rapid_device_error_info(w, clear) != 0) return -1;
    return (int)w[0];
}

rapid_status rapid_stream_status(void* stream, int clear) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        (void)cudaGetLastError();
        return RAPID_ECUDA;
    }
    uint32_t w[8];
    if (rapid_device_error_info(w, clear) != 0) return RAPID_ECUDA;
    if (w[0] & kErrWaitTimeout) return RAPID_ETIMEOUT;
    if (w[0] & kErrBadInput) return RAPID_EINVAL;
    return RAPID_OK;
}

rapid_status rapid_wait_selftest(uint64_t limit_ns, void* stream) {
    if (limit_ns < 1000) limit_ns = 1000;
    if (limit_ns > kWaitLimitNs) limit_ns = kWaitLimitNs;
    unsigned int* err = device_error_word();
    if (!err) return RAPID_ECUDA;
    wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, limit_ns);
    return cudaGetLastError() == cudaSuccess ? RAPID_OK : RAPID_ECUDA;
}

int rapid_device_error_info(uint32_t* words8, int clear) {
    unsigned int v[8];
    if (cudaMemcpyFromSymbol(v, g_device_error, sizeof(v)) != cudaSuccess) return -1;
    if (clear) {
        const unsigned int zero[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (cudaMemcpyToSymbol(g_device_error, zero, sizeof(zero)) != cudaSuccess) return -1;
    }
    if (words8)
        for (int i = 0; i < 8; ++i) words8[i] = v[i];
    return 0;
}

}  // extern "C"
