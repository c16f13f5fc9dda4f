/*
 * rapid.h - C ABI of librapid.so: the long-context verification step of
 * retrieval-augmented speculative decoding on one GB300 (sm_103a).
 *
 * Two operations make up the step:
 *
 *   rapid_verify_attn  attention of the n_q = gamma+1 draft/query tokens of a
 *                      verify pass against a long GQA KV cache, computed as
 *                      "hybrid tree attention": an unmasked pass over the
 *                      history (prefix) rows, a masked pass over the n_q
 *                      speculative rows, and an exact log-sum-exp merge of the
 *                      two partial results.
 *                      Source: "LongSpec: Long-Context Lossless Speculative
 *                      Decoding with Efficient Drafting and Verification",
 *                      section 2.3 (Fast Tree Attention / Hybrid Tree
 *                      Attention): history part without a mask, speculative
 *                      part with a mask, parts combined by log-sum-exp.
 *
 *   rapid_accept       the retrieval-augmented acceptance step over the full
 *                      vocabulary.  Source: "RAPID: Long-Context Inference
 *                      with Retrieval-Augmented Speculative Decoding" (blog
 *                      summary), section 2.1 (speculative-decoding ratio test
 *                      and residual distribution) and section 2.4 (the
 *                      retrieval-augmented target p_hat = softmax(z/T +
 *                      eta*(q - p)), the tail-preserving replacement of p_hat
 *                      by p where p_hat < 0.1 * max p_hat, and the adjusted
 *                      residual norm(max(p - p_hat, p - q))).
 *                      rapid_accept_ex adds drafts of different lengths in
 *                      one batch and a Philox key in device memory (CUDA-graph
 *                      replays); rapid_accept_noalloc needs no workspace.
 *
 *   rapid_attn_merge   the log-sum-exp combine of attention parts computed
 *                      separately (shards of the key range, other devices).
 *
 *   rapid_kv_commit    after acceptance, the accepted path's speculative K/V
 *   rapid_kv_advance   rows join the history next to the root, and the
 *                      history lengths grow by 1 + n_accepted.
 *
 *   rapid_lm_head      the target's logits of the verify rows from the shared
 *   rapid_lm_head_accept  LM head, alone or followed by rapid_accept (or, with
 *                      rapid_lm_head_accept_ex, by rapid_accept_ex).
 *
 *   rapid_retrieval_scores  cosine scores of chunk embeddings against the
 *   rapid_retrieval_select  query, and the budgeted, thresholded choice of
 *                      chunks for the draft's retrieved context ("RAPID ...",
 *                      section 3.1, RAG settings).
 *
 * Conventions shared by every call:
 *  - All tensor arguments are DEVICE pointers owned by the caller.  The library
 *    allocates nothing on these paths; scratch space is the caller's
 *    `workspace` (size from the matching *_workspace_size call, 256-byte
 *    aligned).  Only rapid_kv_commit writes to the KV cache.
 *  - Calls are asynchronous and stream-ordered on `stream` (a cudaStream_t
 *    passed as void*; NULL = the legacy default stream).  No call
 *    synchronises the device; results are valid once the stream reaches them.
 *  - Argument checks that need only host-visible values run before any launch
 *    and return RAPID_EINVAL.  Values that live in device memory (prefix
 *    lengths, token ids, parent pointers, node counts) cannot be checked
 *    without synchronising, so the kernels check them as they run: an
 *    out-of-range value is clamped (or, for a token id, treated as rejected)
 *    so that every memory access stays in bounds, the results of that call are
 *    unspecified, and bit 1 of the device error word is set.
 *    rapid_stream_status turns that bit into RAPID_EINVAL, and a bounded wait
 *    that gave up (bit 0) into RAPID_ETIMEOUT.
 *  - No C++ exception crosses this ABI.  Calls are stateless and may be issued
 *    from several host threads on different streams.
 *  - Every per-step quantity that changes between verify steps (history
 *    lengths, paths, counts, and with rapid_accept_ex the Philox key)
 *    is read from device memory, so one step can be captured in a CUDA graph
 *    and replayed; make a call once outside the capture first (the first call
 *    of a shape sets kernel attributes and looks up driver entry points).
 */
#ifndef RAPID_H
#define RAPID_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RAPID_OK = 0,
    RAPID_EINVAL = -1,      /* bad argument (host-checkable), or, from
                               rapid_stream_status, a bad device-side input */
    RAPID_ECUDA = -2,       /* a CUDA runtime call or kernel launch failed   */
    RAPID_ENOMEM = -3,      /* workspace smaller than the *_workspace_size   */
    RAPID_ETIMEOUT = -4,    /* a bounded wait inside a kernel gave up (from
                               rapid_stream_status): outputs are invalid     */
    RAPID_EUNSUPPORTED = -5 /* shape outside the compiled kernels' limits    */
} rapid_status;

/* Element types of Q, K, V and O. */
enum { RAPID_DTYPE_F32 = 0, RAPID_DTYPE_BF16 = 1 };

/* Flags of rapid_accept. */
enum {
    /* Keep p where p_hat < 0.1 * max(p_hat) ("retrieval-augmented target
     * distribution" section: the tail of p_hat is replaced by the tail of p).
     * Set by default in the Python binding; clear it for the plain p_hat. */
    RAPID_ACCEPT_TAIL_CLAMP = 1u
};

/* Largest sizes the compiled kernels accept. */
enum {
    RAPID_MAX_NQ = 64,        /* query (draft) tokens per sequence            */
    RAPID_MAX_VOCAB = 229376  /* vocabulary entries per row (16 x 14336)      */
};

/* ------------------------------------------------------------------------ */
/* Verify attention                                                          */
/* ------------------------------------------------------------------------ */

/*
 * Bytes of scratch that rapid_verify_attn needs for these sizes.  Returns 0
 * for sizes that rapid_verify_attn would reject.
 */
size_t rapid_verify_attn_workspace_size(int B, int Hq, int Hkv, int d, int n_q,
                                        int64_t kv_capacity, int dtype);

/*
 * O, LSE = attention of the verify queries against the KV cache.
 *
 *  Q          [B, Hq, n_q, d]          dtype; already rotated (RoPE applied).
 *  Kcache     [B, Hkv, kv_capacity, d] dtype; key rows, head-major.
 *  Vcache     [B, Hkv, kv_capacity, d] dtype; value rows, head-major.
 *  dtype      RAPID_DTYPE_BF16 or RAPID_DTYPE_F32 (all of Q, K, V, O).
 *  d          head dimension: 64 or 128.
 *  n_q        query tokens per sequence, 1..RAPID_MAX_NQ.  Query head h uses
 *             KV head h / (Hq / Hkv) (grouped-query attention).
 *  prefix_len device int32 [B]: history rows of sequence b are
 *             [0, prefix_len[b]); its n_q speculative rows are
 *             [prefix_len[b], prefix_len[b] + n_q).  Needs
 *             0 <= prefix_len[b] <= kv_capacity - n_q (else the kernels clamp
 *             it and set bit 1 of the device error word).
 *  spec_mask  device uint8 [B, n_q, n_q] or NULL.  Query i of sequence b sees
 *             speculative row j iff spec_mask[b][i][j] != 0 (a token tree's
 *             ancestor-or-self mask).  NULL means the causal chain j <= i.
 *             Every history row is visible to every query (no mask there).
 *             A query that sees no row at all (no history, mask row all
 *             zero) gets O = 0 and LSE = -inf.
 *  softmax_scale  score multiplier; <= 0 selects 1/sqrt(d).
 *  O          [B, Hq, n_q, d] dtype: softmax-weighted sum of the visible V rows.
 *  LSE        float [B, Hq, n_q]: natural-log log-sum-exp of the scaled scores
 *             over the visible rows.
 *  workspace  device scratch of at least rapid_verify_attn_workspace_size()
 *             bytes, 256-byte aligned; contents need no initialisation.
 *
 * Errors: RAPID_EINVAL for NULL tensors, d not in {64,128}, Hq % Hkv != 0,
 * n_q outside [1, RAPID_MAX_NQ], B < 1, B * Hkv > 65535, kv_capacity < n_q, misaligned
 * pointers (16 bytes); RAPID_ENOMEM for a short workspace; RAPID_ECUDA when a
 * launch fails.
 */
rapid_status rapid_verify_attn(const void* Q, const void* Kcache, const void* Vcache,
                               int dtype, int B, int Hq, int Hkv, int d, int n_q,
                               int64_t kv_capacity, const int32_t* prefix_len,
                               const uint8_t* spec_mask, float softmax_scale,
                               void* O, float* LSE, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * Log-sum-exp merge of attention results computed separately over disjoint
 * key sets: the combine step of hybrid tree attention ("LongSpec ...",
 * section 2.3: the history part and the speculative part are combined
 * through their log-sum-exp), for any number of parts.  With L_p the LSE and
 * O_p the normalised output of part p:
 *     LSE = ln sum_p exp(L_p),   O = sum_p exp(L_p - LSE) O_p.
 * rapid_verify_attn does this for its own splits; this call merges results
 * produced elsewhere, for example the shards of a history split by key range
 * (each shard a rapid_verify_attn call on its rows, the speculative rows
 * visible in exactly one of them: an all-zero spec_mask hides them from the
 * others), possibly computed on other devices and copied here.
 *
 *  O_parts    device [n_parts, rows, d] of dtype: each part's O, rows
 *             flattened (a rapid_verify_attn output is [B, Hq, n_q, d]:
 *             rows = B * Hq * n_q).
 *  LSE_parts  device float [n_parts, rows]: each part's natural-log LSE,
 *             finite or -inf (-inf: the part saw no key for that row; its O
 *             is not read).
 *  dtype      RAPID_DTYPE_BF16 or RAPID_DTYPE_F32 (O_parts and O).
 *  d          64 or 128.
 *  O, LSE     device outputs [rows, d] of dtype and float [rows].  A row with
 *             no finite part gets O = 0, LSE = -inf.
 *
 * Arithmetic in fp32.  Errors: RAPID_EINVAL for NULL pointers, n_parts < 1,
 * rows < 1 or above 2^36, d not 64 or 128, a bad dtype, O_parts or O not
 * 16-byte aligned, LSE arrays not 4-byte aligned; RAPID_ECUDA when the
 * launch fails.
 */
rapid_status rapid_attn_merge(const void* O_parts, const float* LSE_parts, int dtype,
                              int n_parts, int64_t rows, int d, void* O, float* LSE,
                              void* stream);

/* ------------------------------------------------------------------------ */
/* Acceptance                                                                */
/* ------------------------------------------------------------------------ */

/* Bytes of scratch that rapid_accept needs (20 per node of the B * n_q nodes,
 * plus alignment); 0 for rejected sizes. */
size_t rapid_accept_workspace_size(int B, int n_q, int V);

/*
 * Retrieval-augmented acceptance of one verify step.
 *
 *  z_target     device float [B, n_q, V]: target logits.  Row j of sequence b
 *               is the target's next-token distribution after node j (node 0
 *               is the last committed token, nodes 1..n_q-1 are drafts).
 *  q_draft      device float [B, n_q, V]: draft probabilities for the same
 *               rows (rows sum to 1; taken as given, T does not touch them).
 *  draft_tokens device int32 [B, n_q]: token of node i (entry 0 unused).
 *  parent       device int32 [B, n_q] or NULL.  NULL = chain (parent of node
 *               i is i-1).  Otherwise parent[b][i] in [0, i) for i >= 1 gives
 *               a token tree; entry 0 is unused.  A parent outside [0, i) is
 *               clamped into it and a draft token outside [0, V) counts as
 *               rejected; both set bit 1 of the device error word.
 *  T            temperature > 0; eta >= 0 and finite (knowledge-transfer
 *               strength of the retrieval-augmented target).
 *  philox_seed  key of the Philox4x32-10 stream.  Node i of sequence b uses
 *               block (counter = {i, b, 0, 0}, key = {seed & 0xffffffff,
 *               seed >> 32}); word 0 gives r_i (ratio test of node i), word 1
 *               gives u_i.  A uniform is (word >> 8) * 2^-24.
 *  flags        RAPID_ACCEPT_TAIL_CLAMP or 0.
 *
 * Per row j:  p = softmax(z_j / T);  p_hat = softmax(z_j / T + eta (q_j - p));
 * with the tail clamp, p_hat_k := p_k wherever p_hat_k < 0.1 * max p_hat.
 * Node i >= 1 is accepted iff r_i <= min(1, p_hat_j(t_i) / q_j(t_i)) with
 * j = parent(i) (q_j(t_i) = 0 accepts).  For a chain, acceptance stops at the
 * first rejected node; for a tree, every root-to-leaf path is checked the same
 * way and the path with the most accepted nodes wins (ties: smallest leaf
 * index).  Let e be the last accepted node of the winning path (0 if none).
 * The next token is drawn from row e by inverse CDF in token-id order with
 * uniform u_{e+1}: from norm(max(p - p_hat, p - q, 0)) if node e has children
 * (a rejection happened below it; p itself if that residual has zero mass),
 * else from p (the bonus token after a fully accepted path).
 *
 * Outputs (device):  n_accepted int32 [B] (accepted draft nodes, 0..depth),
 * next_token int32 [B], path int32 [B, n_q] or NULL (node ids of the
 * accepted nodes in root-to-leaf order, then -1), diag float [B, n_q, 5] or
 * NULL (for node i >= 1: p_j(t_i), clamped p_hat_j(t_i), q_j(t_i), ratio, r_i;
 * node 0 gets zeros).
 *
 * Errors: RAPID_EINVAL for NULL required tensors, B outside [1, 65535], n_q outside
 * [1, RAPID_MAX_NQ], V outside [1, RAPID_MAX_VOCAB], T <= 0 or not finite,
 * eta < 0 or not finite; RAPID_ENOMEM for a short workspace; RAPID_ECUDA when
 * a launch fails.
 */
rapid_status rapid_accept(const float* z_target, const float* q_draft,
                          const int32_t* draft_tokens, const int32_t* parent,
                          int B, int n_q, int V, float T, float eta,
                          uint64_t philox_seed, uint32_t flags,
                          int32_t* n_accepted, int32_t* next_token, int32_t* path,
                          float* diag, void* workspace, size_t workspace_bytes,
                          void* stream);

/*
 * rapid_accept with two optional inputs in device memory: per-sequence node
 * counts (drafts of different lengths in one batch) and the Philox key.
 *
 *  n_nodes          device int32 [B], 4-byte aligned, or NULL.  Sequence b has
 *                   n_nodes[b] nodes, 1 <= n_nodes[b] <= n_q: node 0 (the
 *                   root) and n_nodes[b] - 1 drafts, a chain or a tree as
 *                   `parent` says.  n_accepted, next_token and path of sequence
 *                   b are those of the same call on its first n_nodes[b] nodes
 *                   alone: the nodes past the count are nobody's children and
 *                   on no path, so a fully accepted short chain ends with the
 *                   bonus draw from p of its last row.  The buffers keep the
 *                   [B, n_q, ...] layout; the padding rows of z_target and
 *                   q_draft are not read, the padding tokens and parents
 *                   (any values) affect no result, and the padding diag
 *                   entries are unspecified.  Counts outside
 *                   [1, n_q] are clamped.  NULL: every sequence has n_q nodes.
 *  philox_seed_dev  device address of one uint64_t, 8-byte aligned, or NULL.
 *                   If given, the kernels read the key from there when they
 *                   run (philox_seed is ignored), so a call captured once in a
 *                   CUDA graph draws fresh numbers on every replay as long as
 *                   the caller changes the value between replays (a kernel or
 *                   a copy of its own inside the same graph).  The call does
 *                   not write it.
 *
 * Every other argument, the results and the errors are those of rapid_accept;
 * a misaligned n_nodes or philox_seed_dev returns RAPID_EINVAL.  With both
 * NULL this is rapid_accept.
 */
rapid_status rapid_accept_ex(const float* z_target, const float* q_draft,
                             const int32_t* draft_tokens, const int32_t* parent,
                             const int32_t* n_nodes, int B, int n_q, int V, float T, float eta,
                             uint64_t philox_seed, const uint64_t* philox_seed_dev,
                             uint32_t flags, int32_t* n_accepted, int32_t* next_token,
                             int32_t* path, float* diag, void* workspace,
                             size_t workspace_bytes, void* stream);

/* Largest B * n_q that rapid_accept_noalloc accepts. */
enum { RAPID_NOALLOC_MAX_NODES = 4096 };

/*
 * rapid_accept without a workspace argument, for callers that cannot
 * allocate device memory where they run the acceptance step: a host framework
 * that owns all device memory and gives its plug-ins no allocator, or a
 * latency-critical decode loop that must never call cudaMalloc (it may
 * synchronise the device).  The pages have no counterpart of this entry
 * point; it computes exactly what rapid_accept computes, with the same
 * arguments and outputs.
 *
 * Scratch: a statically allocated device array of 80 KB inside librapid.so,
 * held by every GPU that loads the library until the process exits.  It fits
 * B * n_q <= RAPID_NOALLOC_MAX_NODES; larger sizes return RAPID_EUNSUPPORTED.
 * The call allocates nothing (no cudaMalloc, cudaFree or allocating library
 * routine).  Every call looks up the array's device address on the current
 * device with cudaGetSymbolAddress (which allocates nothing), so a reset
 * device or a re-created context never sees a stale address.  The first
 * lookup on a device may load the library's device code there: make the
 * first call on a device before any stream capture.
 *
 * Concurrency: every call on a device shares the one array, and the array
 * keeps the last call's contents.  Calls whose kernels overlap on the GPU
 * (different streams, or different host threads, without ordering between
 * them) race on it and give wrong results; order such calls, for example on
 * one stream.
 *
 * Errors: those of rapid_accept (RAPID_EINVAL for B < 1 or n_q outside
 * [1, RAPID_MAX_NQ], among others), plus RAPID_EUNSUPPORTED for B * n_q over
 * the limit and RAPID_ECUDA when the array's address cannot be obtained.
 */
rapid_status rapid_accept_noalloc(const float* z_target, const float* q_draft,
                                  const int32_t* draft_tokens, const int32_t* parent,
                                  int B, int n_q, int V, float T, float eta,
                                  uint64_t philox_seed, uint32_t flags,
                                  int32_t* n_accepted, int32_t* next_token, int32_t* path,
                                  float* diag, void* stream);

/* ------------------------------------------------------------------------ */
/* Misc                                                                      */
/* ------------------------------------------------------------------------ */

/* Static, NUL-terminated description of a status code. */
const char* rapid_status_string(int status);

/* Library version as MAJOR * 10000 + MINOR * 100 + PATCH. */
int rapid_version(void);

/*
 * Sticky error bits that kernels of this library raised on the CURRENT device
 * (bit 0: a bounded wait for an asynchronous copy or a peer gave up, so the
 * outputs of that call are invalid; bit 1: a kernel found an invalid
 * device-side input -- a history length, parent, draft token or node count
 * out of range in rapid_verify_attn / rapid_accept*, or an input that
 * rapid_kv_commit, rapid_kv_advance or rapid_retrieval_select refused,
 * leaving that sequence alone).  Synchronises the device to read the word;
 * clears it when `clear` is non-zero.  Returns -1 if the word could not be
 * read.
 */
int rapid_device_error(int clear);

/*
 * The status of the work issued so far: synchronises `stream`, then reads the
 * sticky error word of the current device (the word is per device, not per
 * stream) and clears it when `clear` is non-zero.  Returns RAPID_ETIMEOUT if
 * a bounded wait inside a kernel gave up (the outputs of that call are
 * invalid), else RAPID_EINVAL if a kernel found an out-of-range device-side
 * input, else RAPID_OK; RAPID_ECUDA if the synchronisation or the read
 * failed (a sticky CUDA error, for instance).
 */
rapid_status rapid_stream_status(void* stream, int clear);

/*
 * Self-test of the bounded waits that every kernel of this library uses on
 * its mbarriers: one small kernel starts a bulk copy, then waits on a barrier
 * phase that nothing completes.  After `limit_ns` nanoseconds (clamped to
 * [1000, 1e9]) the wait gives up, records bit 0 and the code 0xC7000001 in
 * the device error record (rapid_device_error_info), waits for its copy to
 * land and returns, exactly as a kernel whose producer stalled would.  A
 * following rapid_stream_status returns RAPID_ETIMEOUT.  The library has no
 * other way to make a wait run out on purpose; no fault is involved.
 * Errors: RAPID_ECUDA when the launch fails.
 */
rapid_status rapid_wait_selftest(uint64_t limit_ns, void* stream);

/*
 * The full error record of the current device: words8[0] = the sticky bits of
 * rapid_device_error, words8[1] = 0x80000000 | code of the first wait that
 * gave up (which kernel role, which barrier, which tile), words8[2..7]
 * reserved.  Synchronises; clears the record when `clear` is non-zero.
 * Returns 0 on success, -1 if the record could not be read.
 */
int rapid_device_error_info(uint32_t* words8, int clear);

/* ------------------------------------------------------------------------ */
/* KV commit after acceptance                                                */
/* ------------------------------------------------------------------------ */

/* Most layers one rapid_kv_commit call takes. */
enum { RAPID_COMMIT_MAX_LAYERS = 128 };

/*
 * Keep the accepted speculative K/V rows of a verify step and drop the rest.
 * In the verify pass the n_q tokens of a step sit after the history of every
 * layer's cache, node i at row P_b + i with node 0 the root ("LongSpec:
 * Long-Context Lossless Speculative Decoding with Efficient Drafting and
 * Verification", section 2.3, the hybrid tree attention layout).  After
 * acceptance the accepted path's rows, already computed by the verify pass,
 * join the history right after the root, in path order:
 *
 *   K[b, h, P_b + 1 + k, :] := K[b, h, P_b + path[b][k], :]   for k < n_accepted[b]
 *
 * and the same for V, for every KV head h of every layer.  Rows past
 * P_b + n_accepted[b] are left as they are (the next step overwrites them).
 * A chain's path is 1, 2, ..., so nothing moves.  Call rapid_kv_advance after
 * the last layer to grow the history lengths.
 *
 *  K_layers, V_layers  HOST arrays of `layers` device pointers; layer l's
 *                      caches are [B, Hkv, kv_capacity, d] of dtype
 *                      (RAPID_DTYPE_F32 or RAPID_DTYPE_BF16), 16-byte aligned.
 *  prefix_len          device int32 [B]: P_b, the history length before the
 *                      step (the root's row).
 *  path, n_accepted    device int32 [B, n_q] and [B], as rapid_accept writes
 *                      them: the accepted node ids in root-to-leaf order.
 *
 * Sources are read before destinations are written, so overlapping moves
 * (path 2, 3, ...) are safe.  Errors: RAPID_EINVAL for NULL pointers, layers
 * outside [1, RAPID_COMMIT_MAX_LAYERS], B < 1, Hkv < 1, d not 64 or 128, n_q
 * outside [1, RAPID_MAX_NQ], kv_capacity < 1, a bad dtype or unaligned caches;
 * RAPID_ECUDA when the launch fails.  A sequence whose device inputs are
 * invalid (n_accepted outside [0, n_q - 1], P_b + n_q > kv_capacity, a path
 * entry outside [k + 1, n_q - 1] or not increasing) is left untouched and bit
 * 1 of the device error word is set.
 */
rapid_status rapid_kv_commit(void* const* K_layers, void* const* V_layers, int layers, int dtype,
                             int B, int Hkv, int d, int64_t kv_capacity, int n_q,
                             const int32_t* prefix_len, const int32_t* path,
                             const int32_t* n_accepted, void* stream);

/*
 * prefix_len[b] += 1 + n_accepted[b] on the device (the root and the accepted
 * drafts join the history).  A sequence whose n_accepted is outside
 * [0, n_q - 1] or whose P_b + n_q exceeds kv_capacity keeps its length and
 * sets bit 1 of the device error word.  Errors: RAPID_EINVAL for NULL
 * pointers, B < 1, n_q outside [1, RAPID_MAX_NQ], kv_capacity < 1;
 * RAPID_ECUDA on launch failure.
 */
rapid_status rapid_kv_advance(int32_t* prefix_len, const int32_t* n_accepted, int B, int n_q,
                              int64_t kv_capacity, void* stream);

/* ------------------------------------------------------------------------ */
/* Retrieval for the draft's compressed context                              */
/* ------------------------------------------------------------------------ */

/* Most chunks per sequence rapid_retrieval_select takes. */
enum { RAPID_RETRIEVAL_MAX_CHUNKS = 8192 };

/*
 * Cosine similarity of every chunk embedding with its sequence's query
 * embedding ("RAPID: Long-Context Inference with Retrieval-Augmented
 * Speculative Decoding", section 3.1, RAG settings: the context is cut into
 * chunks, each embedded, and chunks are ranked by cosine similarity with the
 * query embedding):
 *   scores[b][j] = <query[b], chunks[b][j]> / (|query[b]| |chunks[b][j]|)
 * (0 when either vector is zero), in fp32.
 *
 *  query   device [B, D], chunks device [B, N, D], both of dtype
 *          RAPID_DTYPE_F32 or RAPID_DTYPE_BF16, 16-byte aligned; D a
 *          multiple of 8 in [8, 8192].
 *  scores  device float [B, N].
 * Errors: RAPID_EINVAL for NULL pointers, B < 1, N < 1, a bad D, dtype or
 * alignment; RAPID_ECUDA on launch failure.
 */
rapid_status rapid_retrieval_scores(const void* query, const void* chunks, int dtype, int B, int N,
                                    int D, float* scores, void* stream);

/*
 * The retrieved context of every sequence from its chunk scores (same
 * section: chunks scoring below `threshold` (0.3 there) are dropped and the
 * retrieved context stays within at least `min_tokens` (4096) tokens and
 * 1 / `ratio` (1/24) of the input).  Reading: sequence b has n_b =
 * context_tokens[b] tokens in ceil(n_b / chunk_tokens) chunks (chunk j holds
 * min(chunk_tokens, n_b - j chunk_tokens)); its budget is max(min_tokens,
 * n_b / ratio); chunks are visited in descending score (ties: lower index),
 * the visit stops at the first chunk below the threshold, and a chunk is kept
 * if its tokens fit what is left of the budget.
 *
 *  scores          device float [B, N] (entries past the sequence's chunk
 *                  count are ignored)
 *  context_tokens  device int32 [B]
 *  selected        device int32 [B, N]: the kept chunk ids in ascending
 *                  order, then -1
 *  n_selected, tokens_selected  device int32 [B]
 * Errors: RAPID_EINVAL for NULL pointers, B < 1, N outside [1,
 * RAPID_RETRIEVAL_MAX_CHUNKS], chunk_tokens < 1, ratio < 1, min_tokens < 0;
 * RAPID_ECUDA on launch failure.  A sequence whose context_tokens is negative
 * or needs more than N chunks keeps nothing and sets bit 1 of the device
 * error word.
 */
rapid_status rapid_retrieval_select(const float* scores, const int32_t* context_tokens, int B, int N,
                                    int chunk_tokens, float threshold, int min_tokens, int ratio,
                                    int32_t* selected, int32_t* n_selected,
                                    int32_t* tokens_selected, void* stream);
/* ------------------------------------------------------------------------ */
/* Target logits from the shared LM head                                     */
/* ------------------------------------------------------------------------ */

/* Limits of rapid_lm_head (rows = verify rows of one call). */
enum {
    RAPID_LM_HEAD_MAX_ROWS = 256,
    RAPID_LM_HEAD_MAX_HIDDEN = 16384,
    RAPID_LM_HEAD_MAX_VOCAB = 1 << 22
};

/*
 * The target's logits of the verify rows from their final hidden states and
 * the LM head ("LongSpec: Long-Context Lossless Speculative Decoding with
 * Efficient Drafting and Verification", section 2.1: the drafter shares the
 * target's embedding and LM-head weights; "RAPID: Long-Context Inference with
 * Retrieval-Augmented Speculative Decoding", section 2.1: z is the target's
 * logit vector over the vocabulary):
 *   z[r][v] = sum_k hidden[r][k] * W_lm[v][k],   fp32 accumulation.
 *
 *  hidden  device bf16 [rows, hidden_dim], 16-byte aligned
 *  W_lm    device bf16 [V, hidden_dim] (one vocabulary entry per row, the
 *          usual LM-head weight layout), 16-byte aligned
 *  z       device fp32 [rows, V]
 * rows in [1, RAPID_LM_HEAD_MAX_ROWS]; hidden_dim a multiple of 64 in [64,
 * RAPID_LM_HEAD_MAX_HIDDEN]; V in [1, RAPID_LM_HEAD_MAX_VOCAB].
 * Errors: RAPID_EINVAL for NULL pointers, sizes out of range or misaligned
 * pointers; RAPID_EUNSUPPORTED without the driver's tensor-map encoder;
 * RAPID_ECUDA on launch failure.  A bounded wait inside the kernel that runs
 * out (one second) sets bit 0 of the device error word; z is then invalid.
 */
rapid_status rapid_lm_head(const void* hidden, const void* W_lm, int rows, int hidden_dim, int V,
                           float* z, void* stream);

/* Bytes of scratch that rapid_lm_head_accept needs: the B * n_q * V fp32
 * logits plus rapid_accept's scratch; 0 for unsupported sizes. */
size_t rapid_lm_head_accept_workspace_size(int B, int n_q, int V);

/*
 * rapid_accept on logits that rapid_lm_head computes from the verify rows'
 * hidden states [B * n_q, hidden_dim] (row b * n_q + i is node i of sequence
 * b); the caller never holds the logits.
 *
 * Up to 16 rows (one verify step of an 11-node chain or a 16-node tree), V a
 * multiple of 4 and q_draft 16-byte aligned: ONE cooperative kernel, one CTA
 * per SM, computes the product and then the acceptance step itself.  Each CTA
 * keeps its run of the vocabulary of z in shared memory (z is never written
 * to memory) with the same run of q beside it; the vocabulary-wide softmax
 * statistics, the ratio tests, the path choice and the residual draw follow,
 * with one grid-wide barrier after each of the three vocabulary-wide
 * reductions.  The call first zeroes a 4-byte barrier counter at the front of
 * the workspace (a memset on `stream`); calls on one workspace must not
 * overlap.  The arithmetic is rapid_accept's up to the order of fp32 sums, so
 * probabilities agree with rapid_accept's to about 1e-6 relative and
 * decisions agree except at the near-boundary cases of the ratio test, the
 * tail threshold and the inverse CDF.
 *
 * Otherwise (more rows, or a device without cooperative launches) two
 * launches run back to back on `stream`: rapid_lm_head into the workspace
 * (11 x 128256 fp32 = 5.6 MB for one step, which stays in L2), then
 * rapid_accept on it.
 *
 * Every other argument, output and error is rapid_accept's; B * n_q is at
 * most RAPID_LM_HEAD_MAX_ROWS and V at most RAPID_MAX_VOCAB.
 */
rapid_status rapid_lm_head_accept(const void* hidden, const void* W_lm, int hidden_dim,
                                  const float* q_draft, const int32_t* draft_tokens,
                                  const int32_t* parent, int B, int n_q, int V, float T, float eta,
                                  uint64_t philox_seed, uint32_t flags, int32_t* n_accepted,
                                  int32_t* next_token, int32_t* path, float* diag,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * rapid_lm_head_accept with rapid_accept_ex's two optional device inputs:
 * per-sequence node counts n_nodes (the logits of every row are still
 * computed) and the Philox key at philox_seed_dev.  Same workspace size as
 * rapid_lm_head_accept; the errors of both calls.
 */
rapid_status rapid_lm_head_accept_ex(const void* hidden, const void* W_lm, int hidden_dim,
                                     const float* q_draft, const int32_t* draft_tokens,
                                     const int32_t* parent, const int32_t* n_nodes, int B,
                                     int n_q, int V, float T, float eta, uint64_t philox_seed,
                                     const uint64_t* philox_seed_dev, uint32_t flags,
                                     int32_t* n_accepted, int32_t* next_token, int32_t* path,
                                     float* diag, void* workspace, size_t workspace_bytes,
                                     void* stream);


#ifdef __cplusplus
}
#endif

#endif /* RAPID_H */
