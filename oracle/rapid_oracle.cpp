/*
 * TEST INFRASTRUCTURE -- plain double-precision CPU oracle of the verification
 * step of retrieval-augmented speculative decoding.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline / reference
 * arm may load this library.  The product (librapid.so and its Python binding)
 * never links, imports or calls it, and it shares no code with the CUDA path:
 * its Philox generator, its bf16 decoding and every formula below are written
 * here independently, straight from the definitions they cite.
 *
 * Sources (page title, then section / equation):
 *  [RAPID]    "RAPID: Long-Context Inference with Retrieval-Augmented
 *             Speculative Decoding" (blog summary).  Section 2.1: the
 *             speculative-decoding ratio test r <= min(1, p(x')/q(x')) with
 *             r ~ U(0,1) and the residual norm(max(p - q, 0)).  Section 2.4:
 *             Eq. (4) p_hat = softmax(z/T + eta (q - p)); Proposition 1
 *             (d/dz of T^2 KL(q || p) is T (p - q)); the distilled logit
 *             z_hat = z + eta T (q - p); the tail rule p_hat_k := p_k where
 *             p_hat_k < 0.1 max_j p_hat_j; the adjusted residual
 *             norm(max(p - p_hat, p - q)).
 *  [LongSpec] "LongSpec: Long-Context Lossless Speculative Decoding with
 *             Efficient Drafting and Verification", section 2.3 (Hybrid Tree
 *             Attention): the history part is attended without a mask, the
 *             speculative part with a mask, and the two partial outputs are
 *             combined with the log-sum-exp trick.
 *  [Philox]   Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *             1, 2, 3" (SC'11): the Philox4x32 bijection, 10 rounds.
 *
 * Readings where the pages are silent or garbled (each also listed in the
 * design notes): the tail rule compares against the max of the unclamped
 * p_hat and does not renormalise; the ratio test and the residual use the
 * clamped p_hat; the residual is clipped at 0 before normalising and falls
 * back to p when it has no mass; the bonus token after a fully accepted path
 * is drawn from p; the tree rule checks every root-to-leaf path and keeps the
 * longest accepted prefix (ties: smallest leaf id).
 *
 * Parity of the tree path-selection rule is unpinned beyond brute-force
 * enumeration of tiny trees (the pages define only the tree mask).
 *
 * Retrieval ([RAPID] explainer and paper pages, section 3.1 "RAG settings"):
 * the long context is cut into 512-token chunks, each embedded; a chunk's
 * score is the cosine similarity of its embedding with the query embedding;
 * chunks scoring below 0.3 are dropped and the top ones are kept within a
 * retrieved-context budget of at least 4096 tokens and 1/24 of the input
 * (reading: budget = max(4096, n / 24); chunks taken greedily in descending
 * score, ties to the lower index, a chunk that does not fit the remaining
 * budget is skipped; the kept chunks are returned in document order).
 *
 * KV commit (the step after acceptance; the pages describe the verify pass's
 * cache layout -- [LongSpec] section 2.3, speculative rows after the history,
 * node i of the step at position P + i, node 0 the root -- but print no
 * commit step): the accepted path's rows, already computed by the verify
 * pass, join the history right after the root in path order, and the history
 * length grows by 1 + n_accepted; the other speculative rows are dropped by
 * not counting them.
 */
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

// ----------------------------------------------------------------------------
// Philox4x32-10 [Philox].  Round: two 32x32->64 multiplies with the published
// multipliers; the key is bumped by the published Weyl constants between
// rounds.
// ----------------------------------------------------------------------------
const uint32_t kPhiloxMul0 = 0xD2511F53u;
const uint32_t kPhiloxMul1 = 0xCD9E8D57u;
const uint32_t kPhiloxWeyl0 = 0x9E3779B9u;
const uint32_t kPhiloxWeyl1 = 0xBB67AE85u;

void philox4x32_10(const uint32_t in_ctr[4], const uint32_t in_key[2], uint32_t out[4]) {
    uint32_t c0 = in_ctr[0], c1 = in_ctr[1], c2 = in_ctr[2], c3 = in_ctr[3];
    uint32_t k0 = in_key[0], k1 = in_key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += kPhiloxWeyl0;
            k1 += kPhiloxWeyl1;
        }
        uint64_t prod0 = (uint64_t)kPhiloxMul0 * (uint64_t)c0;
        uint64_t prod1 = (uint64_t)kPhiloxMul1 * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

// A 32-bit word becomes a uniform in [0, 1) from its top 24 bits; the value is
// exact in both float and double.
double word_to_uniform(uint32_t w) { return (double)(w >> 8) * (1.0 / 16777216.0); }

// Node i of sequence b: r_i from word 0, u_i from word 1 of block {i, b, 0, 0}.
void node_uniforms(uint64_t seed, int b, int i, double* r, double* u) {
    uint32_t ctr[4] = {(uint32_t)i, (uint32_t)b, 0u, 0u};
    uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
    uint32_t out[4];
    philox4x32_10(ctr, key, out);
    if (r) *r = word_to_uniform(out[0]);
    if (u) *u = word_to_uniform(out[1]);
}

// ----------------------------------------------------------------------------
// Element decoding: dtype 0 = IEEE float32, 1 = bfloat16 (the upper 16 bits of
// a float32).  Both convert to double exactly.
// ----------------------------------------------------------------------------
double load_elem(const void* base, int64_t idx, int dtype) {
    if (dtype == 0) return (double)((const float*)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
    float f;
    std::memcpy(&f, &bits, sizeof(f));
    return (double)f;
}

struct AttnProblem {
    const void* Q;
    const void* K;
    const void* V;
    int dtype, B, Hq, Hkv, d, n_q;
    int64_t cap;
    const int32_t* prefix_len;
    const uint8_t* mask;  // NULL: causal chain
    double scale;
};

// Is speculative row j visible to query i of sequence b?
bool spec_visible(const AttnProblem& P, int b, int i, int j) {
    if (!P.mask) return j <= i;
    return P.mask[((int64_t)b * P.n_q + i) * P.n_q + j] != 0;
}

// One query row, by the definition of attention: scores of every visible key
// row (all history rows, plus the speculative rows the mask allows), softmax,
// weighted sum of the value rows.  LSE = log sum_j exp(s_j).
void attn_row_plain(const AttnProblem& P, int b, int h, int i, double* out_o, double* out_lse) {
    const int G = P.Hq / P.Hkv;
    const int g = h / G;
    const int d = P.d;
    const int64_t q_off = (((int64_t)b * P.Hq + h) * P.n_q + i) * d;
    const int64_t kv_head = ((int64_t)b * P.Hkv + g) * P.cap;
    const int64_t prefix = P.prefix_len[b];

    std::vector<double> q(d);
    for (int k = 0; k < d; ++k) q[k] = load_elem(P.Q, q_off + k, P.dtype);

    std::vector<int64_t> rows;
    rows.reserve(prefix + P.n_q);
    for (int64_t j = 0; j < prefix; ++j) rows.push_back(j);
    for (int j = 0; j < P.n_q; ++j)
        if (spec_visible(P, b, i, j)) rows.push_back(prefix + j);

    std::vector<double> s(rows.size());
    double m = -std::numeric_limits<double>::infinity();
    for (size_t n = 0; n < rows.size(); ++n) {
        const int64_t base = (kv_head + rows[n]) * d;
        double dot = 0.0;
        for (int k = 0; k < d; ++k) dot += q[k] * load_elem(P.K, base + k, P.dtype);
        s[n] = P.scale * dot;
        m = std::max(m, s[n]);
    }
    double denom = 0.0;
    for (size_t n = 0; n < rows.size(); ++n) denom += std::exp(s[n] - m);
    for (int k = 0; k < d; ++k) out_o[k] = 0.0;
    for (size_t n = 0; n < rows.size(); ++n) {
        const double wgt = std::exp(s[n] - m) / denom;
        const int64_t base = (kv_head + rows[n]) * d;
        for (int k = 0; k < d; ++k) out_o[k] += wgt * load_elem(P.V, base + k, P.dtype);
    }
    *out_lse = m + std::log(denom);
}

// A partial result over a subset of key rows: un-normalised weighted sum with
// its own running max, as the log-sum-exp combination needs.
struct Partial {
    double m = -std::numeric_limits<double>::infinity();
    double l = 0.0;
    std::vector<double> acc;
};

Partial attn_partial(const AttnProblem& P, const std::vector<double>& q, int64_t kv_head,
                     const std::vector<int64_t>& rows) {
    Partial part;
    part.acc.assign(P.d, 0.0);
    std::vector<double> s(rows.size());
    for (size_t n = 0; n < rows.size(); ++n) {
        const int64_t base = (kv_head + rows[n]) * P.d;
        double dot = 0.0;
        for (int k = 0; k < P.d; ++k) dot += q[k] * load_elem(P.K, base + k, P.dtype);
        s[n] = P.scale * dot;
        part.m = std::max(part.m, s[n]);
    }
    for (size_t n = 0; n < rows.size(); ++n) {
        const double e = std::exp(s[n] - part.m);
        part.l += e;
        const int64_t base = (kv_head + rows[n]) * P.d;
        for (int k = 0; k < P.d; ++k) part.acc[k] += e * load_elem(P.V, base + k, P.dtype);
    }
    return part;
}

// The hybrid form [LongSpec 2.3]: the history rows cut at the given
// boundaries into unmasked pieces (empty pieces allowed), the speculative rows
// under the mask as one more piece, every piece normalised on its own, then
// combined by log-sum-exp:  L = log sum_p exp(L_p),  O = sum_p exp(L_p - L) O_p.
void attn_row_split(const AttnProblem& P, int b, int h, int i, const int64_t* cuts, int n_cuts,
                    double* out_o, double* out_lse) {
    const int G = P.Hq / P.Hkv;
    const int g = h / G;
    const int64_t q_off = (((int64_t)b * P.Hq + h) * P.n_q + i) * P.d;
    const int64_t kv_head = ((int64_t)b * P.Hkv + g) * P.cap;
    const int64_t prefix = P.prefix_len[b];
    std::vector<double> q(P.d);
    for (int k = 0; k < P.d; ++k) q[k] = load_elem(P.Q, q_off + k, P.dtype);

    std::vector<Partial> parts;
    int64_t lo = 0;
    for (int c = 0; c <= n_cuts; ++c) {
        int64_t hi = (c < n_cuts) ? std::min<int64_t>(std::max<int64_t>(cuts[c], lo), prefix) : prefix;
        std::vector<int64_t> rows;
        for (int64_t j = lo; j < hi; ++j) rows.push_back(j);
        parts.push_back(attn_partial(P, q, kv_head, rows));
        lo = hi;
    }
    std::vector<int64_t> spec_rows;
    for (int j = 0; j < P.n_q; ++j)
        if (spec_visible(P, b, i, j)) spec_rows.push_back(prefix + j);
    parts.push_back(attn_partial(P, q, kv_head, spec_rows));

    // Per-piece normalised output and LSE; an empty piece has LSE = -inf.
    double L_max = -std::numeric_limits<double>::infinity();
    std::vector<double> lse(parts.size());
    for (size_t p = 0; p < parts.size(); ++p) {
        lse[p] = parts[p].l > 0.0 ? parts[p].m + std::log(parts[p].l)
                                  : -std::numeric_limits<double>::infinity();
        L_max = std::max(L_max, lse[p]);
    }
    double sum = 0.0;
    for (size_t p = 0; p < parts.size(); ++p)
        if (parts[p].l > 0.0) sum += std::exp(lse[p] - L_max);
    const double L = L_max + std::log(sum);
    for (int k = 0; k < P.d; ++k) out_o[k] = 0.0;
    for (size_t p = 0; p < parts.size(); ++p) {
        if (parts[p].l <= 0.0) continue;
        const double wgt = std::exp(lse[p] - L);
        for (int k = 0; k < P.d; ++k) out_o[k] += wgt * (parts[p].acc[k] / parts[p].l);
    }
    *out_lse = L;
}

template <class F>
void parallel_for(int64_t n, int nthreads, F fn) {
    if (nthreads <= 1 || n <= 1) {
        for (int64_t t = 0; t < n; ++t) fn(t);
        return;
    }
    nthreads = (int)std::min<int64_t>(nthreads, n);
    std::vector<std::thread> pool;
    for (int w = 0; w < nthreads; ++w)
        pool.emplace_back([=, &fn]() {
            for (int64_t t = w; t < n; t += nthreads) fn(t);
        });
    for (auto& th : pool) th.join();
}

// ----------------------------------------------------------------------------
// Acceptance [RAPID 2.1, 2.4]
// ----------------------------------------------------------------------------

// p = softmax(z/T); p_hat_raw = softmax(z/T + eta (q - p)); p_hat = p_hat_raw
// with the tail rule (if clamp): p_hat_k := p_k where p_hat_raw_k < 0.1 max p_hat_raw.
void row_dists(const float* z, const float* q, int V, double T, double eta, int clamp,
               double* p, double* phat_raw, double* phat) {
    std::vector<double> x(V), a(V);
    double m1 = -std::numeric_limits<double>::infinity();
    for (int k = 0; k < V; ++k) {
        x[k] = (double)z[k] / T;
        m1 = std::max(m1, x[k]);
    }
    double s1 = 0.0;
    for (int k = 0; k < V; ++k) s1 += std::exp(x[k] - m1);
    for (int k = 0; k < V; ++k) p[k] = std::exp(x[k] - m1) / s1;

    double m2 = -std::numeric_limits<double>::infinity();
    for (int k = 0; k < V; ++k) {
        a[k] = x[k] + eta * ((double)q[k] - p[k]);
        m2 = std::max(m2, a[k]);
    }
    double s2 = 0.0;
    for (int k = 0; k < V; ++k) s2 += std::exp(a[k] - m2);
    for (int k = 0; k < V; ++k) phat_raw[k] = std::exp(a[k] - m2) / s2;

    double top = 0.0;
    for (int k = 0; k < V; ++k) top = std::max(top, phat_raw[k]);
    for (int k = 0; k < V; ++k)
        phat[k] = (clamp && phat_raw[k] < 0.1 * top) ? p[k] : phat_raw[k];
}

// Adjusted residual weights max(p - p_hat, p - q, 0); with eta = 0 and no
// clamp effect this is the plain max(p - q, 0) of section 2.1.
void residual_weights(const double* p, const double* phat, const float* q, int V, double* w) {
    for (int k = 0; k < V; ++k) w[k] = std::max(std::max(p[k] - phat[k], p[k] - (double)q[k]), 0.0);
}

// Inverse CDF in ascending token id: the smallest k with C_k > u * W, where
// C_k = w_0 + ... + w_k and W = C_{V-1}.  If rounding leaves no such k, the
// last token with positive weight.
int sample_inverse_cdf(const double* w, int V, double u, double* W_out, double* target_out) {
    double W = 0.0;
    for (int k = 0; k < V; ++k) W += w[k];
    const double target = u * W;
    if (W_out) *W_out = W;
    if (target_out) *target_out = target;
    double C = 0.0;
    int last_pos = 0;
    for (int k = 0; k < V; ++k) {
        C += w[k];
        if (w[k] > 0.0) last_pos = k;
        if (C > target) return k;
    }
    return last_pos;
}

struct AcceptProblem {
    const float* z;
    const float* q;
    const int32_t* tokens;
    const int32_t* parent;  // NULL: chain
    const int32_t* n_nodes; // NULL: n_q nodes in every sequence
    int B, n_q, V;
    double T, eta;
    uint64_t seed;
    int clamp;
};

int parent_of(const AcceptProblem& A, int b, int i) {
    return A.parent ? A.parent[(int64_t)b * A.n_q + i] : i - 1;
}

// A sequence with n nodes (a draft shorter than the batch's n_q) is the same
// step on its first n nodes alone: only the strides of the [B, n_q, ...]
// arrays still use n_q.  The nodes past n are not looked at.
void accept_one(const AcceptProblem& A, int b, int32_t* n_acc, int32_t* next_tok, int32_t* path,
                double* diag, double* sample_info) {
    const int stride = A.n_q, V = A.V;
    const int n_q = A.n_nodes ? A.n_nodes[b] : A.n_q;   // nodes of this sequence
    const int64_t rowsz = V;
    std::vector<std::vector<double>> P(n_q), PH(n_q);
    std::vector<double> scratch(V);
    if (diag) for (int c = 0; c < stride * 5; ++c) diag[(int64_t)b * stride * 5 + c] = 0.0;
    for (int j = 0; j < n_q; ++j) {
        P[j].resize(V);
        PH[j].resize(V);
        const int64_t off = ((int64_t)b * stride + j) * rowsz;
        row_dists(A.z + off, A.q + off, V, A.T, A.eta, A.clamp, P[j].data(), scratch.data(),
                  PH[j].data());
    }

    // Ratio test of every draft node against its parent's row.
    std::vector<int> accepted(n_q, 0);
    for (int i = 1; i < n_q; ++i) {
        const int j = parent_of(A, b, i);
        const int t = A.tokens[(int64_t)b * stride + i];
        const double pt = P[j][t];
        const double ph = PH[j][t];
        const double qt = (double)A.q[((int64_t)b * stride + j) * rowsz + t];
        const double ratio = (qt == 0.0) ? std::numeric_limits<double>::infinity() : ph / qt;
        double r;
        node_uniforms(A.seed, b, i, &r, nullptr);
        accepted[i] = (r <= std::min(1.0, ratio)) ? 1 : 0;
        if (diag) {
            double* dg = diag + ((int64_t)b * stride + i) * 5;
            dg[0] = pt; dg[1] = ph; dg[2] = qt; dg[3] = ratio; dg[4] = r;
        }
    }

    // Children lists; leaves are nodes without children.
    std::vector<int> n_children(n_q, 0);
    for (int i = 1; i < n_q; ++i) n_children[parent_of(A, b, i)]++;

    // Every root-to-leaf path: count the accepted nodes from the top down to
    // the first rejection.  Keep the longest; on a tie the smallest leaf id.
    int best_len = -1, best_leaf = 0;
    std::vector<int> best_nodes;
    for (int leaf = 0; leaf < n_q; ++leaf) {
        if (n_children[leaf] != 0) continue;
        std::vector<int> nodes;  // leaf ... up to (excluding) the root
        for (int v = leaf; v != 0; v = parent_of(A, b, v)) nodes.push_back(v);
        std::reverse(nodes.begin(), nodes.end());
        int len = 0;
        while (len < (int)nodes.size() && accepted[nodes[len]]) ++len;
        if (len > best_len) {
            best_len = len;
            best_leaf = leaf;
            best_nodes.assign(nodes.begin(), nodes.begin() + len);
        }
    }
    (void)best_leaf;
    const int e = best_len > 0 ? best_nodes[best_len - 1] : 0;

    // Next token from row e with u_{e+1}: the adjusted residual if a rejection
    // happened below e, else the bonus draw from p.
    double u;
    node_uniforms(A.seed, b, e + 1, nullptr, &u);
    std::vector<double> w(V);
    int kind;
    if (n_children[e] > 0) {
        const int64_t off = ((int64_t)b * stride + e) * rowsz;
        residual_weights(P[e].data(), PH[e].data(), A.q + off, V, w.data());
        double W = 0.0;
        for (int k = 0; k < V; ++k) W += w[k];
        if (W > 0.0) {
            kind = 1;
        } else {
            w = P[e];
            kind = 2;
        }
    } else {
        w = P[e];
        kind = 0;
    }
    double W, target;
    const int tok = sample_inverse_cdf(w.data(), V, u, &W, &target);
    n_acc[b] = best_len;
    next_tok[b] = tok;
    if (path) {
        for (int n = 0; n < stride; ++n) path[(int64_t)b * stride + n] = n < best_len ? best_nodes[n] : -1;
    }
    if (sample_info) {
        double* si = sample_info + (int64_t)b * 6;
        si[0] = e; si[1] = kind; si[2] = u; si[3] = W; si[4] = target; si[5] = tok;
    }
}

}  // namespace

extern "C" {

int orc_version(void) { return 1; }

// K, V: [layers, B, Hkv, cap, row_bytes] opaque rows.  For every (layer, b, h)
// and k < n_acc[b]: row P_b + 1 + k takes the row that node path[b][k] had
// (P_b = prefix_len[b]), all sources read before any destination is written.
// A sequence with an invalid input (n_acc outside [0, n_q - 1], P_b < 0,
// P_b + n_q > cap, a path entry outside [k + 1, n_q - 1] or not increasing) is
// left untouched; returns how many sequences were.
int orc_kv_commit(uint8_t* K, uint8_t* V, int layers, int B, int Hkv, int64_t cap, int row_bytes,
                  int n_q, const int32_t* prefix_len, const int32_t* path, const int32_t* n_acc) {
    int bad = 0;
    for (int b = 0; b < B; ++b) {
        const int n = n_acc[b];
        const int64_t P = prefix_len[b];
        bool ok = n >= 0 && n <= n_q - 1 && P >= 0 && P + n_q <= cap;
        for (int k = 0; ok && k < n; ++k) {
            const int src = path[(int64_t)b * n_q + k];
            if (src < k + 1 || src > n_q - 1) ok = false;
            if (k > 0 && src <= path[(int64_t)b * n_q + k - 1]) ok = false;
        }
        if (!ok) {
            ++bad;
            continue;
        }
        std::vector<uint8_t> rows((size_t)n * row_bytes);
        for (int l = 0; l < layers; ++l) {
            for (int h = 0; h < Hkv; ++h) {
                for (uint8_t* cache : {K, V}) {
                    uint8_t* base = cache + ((((int64_t)l * B + b) * Hkv + h) * cap + P) * row_bytes;
                    for (int k = 0; k < n; ++k)
                        std::memcpy(&rows[(size_t)k * row_bytes],
                                    base + (int64_t)path[(int64_t)b * n_q + k] * row_bytes, row_bytes);
                    for (int k = 0; k < n; ++k)
                        std::memcpy(base + (int64_t)(1 + k) * row_bytes, &rows[(size_t)k * row_bytes],
                                    row_bytes);
                }
            }
        }
    }
    return bad;
}

// Cosine similarity of each chunk embedding with its sequence's query
// embedding, in double: s = <q, c> / (|q| |c|), 0 if either vector is zero.
// query [B, D], chunks [B, N, D], both float32.
void orc_retrieval_scores(const float* query, const float* chunks, int B, int N, int D,
                          double* scores) {
    for (int b = 0; b < B; ++b) {
        const float* q = query + (int64_t)b * D;
        double qq = 0.0;
        for (int k = 0; k < D; ++k) qq += (double)q[k] * q[k];
        for (int j = 0; j < N; ++j) {
            const float* c = chunks + ((int64_t)b * N + j) * D;
            double qc = 0.0, cc = 0.0;
            for (int k = 0; k < D; ++k) {
                qc += (double)q[k] * c[k];
                cc += (double)c[k] * c[k];
            }
            scores[(int64_t)b * N + j] = (qq > 0.0 && cc > 0.0) ? qc / (std::sqrt(qq) * std::sqrt(cc)) : 0.0;
        }
    }
}

// The retrieved context of each sequence from its chunk scores (float32, the
// precision the decision is taken in): sequence b has n_b = context_tokens[b]
// tokens in ceil(n_b / chunk) chunks, chunk j holding min(chunk, n_b - j chunk)
// of them; budget_b = max(min_tokens, n_b / ratio).  Chunks are visited in
// descending score (ties: lower index); the visit stops at the first chunk
// below the threshold; a chunk is kept if its tokens fit what is left of the
// budget.  selected[b][0 .. n_sel) = kept chunk ids, ascending.
void orc_retrieval_select(const float* scores, const int32_t* context_tokens, int B, int N,
                          int chunk, float threshold, int min_tokens, int ratio,
                          int32_t* selected, int32_t* n_selected, int32_t* tokens_selected) {
    for (int b = 0; b < B; ++b) {
        const int64_t n = context_tokens[b];
        int nc = (int)((n + chunk - 1) / chunk);
        if (nc > N) nc = N;
        const int64_t budget = std::max<int64_t>(min_tokens, n / ratio);
        std::vector<int> order(nc);
        for (int j = 0; j < nc; ++j) order[j] = j;
        const float* s = scores + (int64_t)b * N;
        std::sort(order.begin(), order.end(), [&](int x, int y) {
            return s[x] > s[y] || (s[x] == s[y] && x < y);
        });
        std::vector<char> keep(nc, 0);
        int64_t left = budget, used = 0;
        int cnt = 0;
        for (int j : order) {
            if (!(s[j] >= threshold)) break;
            const int64_t len = std::min<int64_t>(chunk, n - (int64_t)j * chunk);
            if (len <= left) {
                keep[j] = 1;
                left -= len;
                used += len;
                ++cnt;
            }
        }
        int w = 0;
        for (int j = 0; j < nc; ++j)
            if (keep[j]) selected[(int64_t)b * N + w++] = j;
        for (int j = w; j < N; ++j) selected[(int64_t)b * N + j] = -1;
        n_selected[b] = cnt;
        tokens_selected[b] = (int32_t)used;
    }
}

// Target logits of the verify rows from their final hidden states and the LM
// head ("LongSpec: Long-Context Lossless Speculative Decoding with Efficient
// Drafting and Verification", section 2.1: the drafter and the target share
// the embedding and LM-head weights; "RAPID ..." section 2.1: z is the
// target's logit vector over the vocabulary):
//   z[r][v] = sum_k H[r][k] * W[v][k],
// H [rows, hidden] and W [V, hidden] (one vocabulary entry per row of W, the
// usual LM-head weight layout), summed in double.
void orc_lm_head_logits(const float* H, const float* W, int rows, int hidden, int V, double* z,
                        int nthreads) {
    parallel_for(V, nthreads, [&](int64_t v) {
        const float* w = W + v * hidden;
        for (int r = 0; r < rows; ++r) {
            const float* h = H + (int64_t)r * hidden;
            double acc = 0.0;
            for (int k = 0; k < hidden; ++k) acc += (double)h[k] * (double)w[k];
            z[(int64_t)r * V + v] = acc;
        }
    });
}

// The history after a committed step: the root and the accepted rows join it.
void orc_kv_advance(int32_t* prefix_len, const int32_t* n_acc, int B) {
    for (int b = 0; b < B; ++b) prefix_len[b] += 1 + n_acc[b];
}

void orc_philox4x32_10(const uint32_t* ctr, const uint32_t* key, uint32_t* out) {
    philox4x32_10(ctr, key, out);
}

void orc_node_uniforms(uint64_t seed, int b, int i, double* r, double* u) {
    node_uniforms(seed, b, i, r, u);
}

// Full attention by the definition; O [B,Hq,n_q,d], LSE [B,Hq,n_q] in double.
void orc_verify_attn(const void* Q, const void* K, const void* V, int dtype, int B, int Hq, int Hkv,
                     int d, int n_q, int64_t cap, const int32_t* prefix_len, const uint8_t* mask,
                     double scale, double* O, double* LSE, int nthreads) {
    AttnProblem P{Q, K, V, dtype, B, Hq, Hkv, d, n_q, cap, prefix_len, mask, scale};
    const int64_t rows = (int64_t)B * Hq * n_q;
    parallel_for(rows, nthreads, [&](int64_t r) {
        const int i = (int)(r % n_q);
        const int h = (int)((r / n_q) % Hq);
        const int b = (int)(r / ((int64_t)n_q * Hq));
        attn_row_plain(P, b, h, i, O + r * d, LSE + r);
    });
}

// Selected rows only (b, h, i triples), for spot checks at full size.
void orc_verify_attn_rows(const void* Q, const void* K, const void* V, int dtype, int B, int Hq,
                          int Hkv, int d, int n_q, int64_t cap, const int32_t* prefix_len,
                          const uint8_t* mask, double scale, const int32_t* bhi, int n_rows,
                          double* O, double* LSE, int nthreads) {
    AttnProblem P{Q, K, V, dtype, B, Hq, Hkv, d, n_q, cap, prefix_len, mask, scale};
    parallel_for(n_rows, nthreads, [&](int64_t r) {
        attn_row_plain(P, bhi[3 * r], bhi[3 * r + 1], bhi[3 * r + 2], O + r * d, LSE + r);
    });
}

// Hybrid form: history cut at cuts[0..n_cuts), speculative piece, LSE merge.
void orc_verify_attn_split(const void* Q, const void* K, const void* V, int dtype, int B, int Hq,
                           int Hkv, int d, int n_q, int64_t cap, const int32_t* prefix_len,
                           const uint8_t* mask, double scale, const int64_t* cuts, int n_cuts,
                           double* O, double* LSE, int nthreads) {
    AttnProblem P{Q, K, V, dtype, B, Hq, Hkv, d, n_q, cap, prefix_len, mask, scale};
    const int64_t rows = (int64_t)B * Hq * n_q;
    parallel_for(rows, nthreads, [&](int64_t r) {
        const int i = (int)(r % n_q);
        const int h = (int)((r / n_q) % Hq);
        const int b = (int)(r / ((int64_t)n_q * Hq));
        attn_row_split(P, b, h, i, cuts, n_cuts, O + r * d, LSE + r);
    });
}

// Log-sum-exp combine of parts computed over disjoint key sets ("LongSpec",
// section 2.3, Hybrid Tree Attention: parts combined through their
// log-sum-exp), written out for any number of parts: LSE = ln sum_p
// exp(LSE_p), O = sum_p exp(LSE_p - LSE) O_p.  Parts with LSE_p = -inf saw
// no key and add nothing; a row with no such part gets O = 0, LSE = -inf.
void orc_lse_merge(const double* O_parts, const double* LSE_parts, int n_parts, int64_t rows,
                   int d, double* O, double* LSE) {
    const double ninf = -std::numeric_limits<double>::infinity();
    for (int64_t r = 0; r < rows; ++r) {
        double m = ninf;
        for (int p = 0; p < n_parts; ++p) m = std::max(m, LSE_parts[(int64_t)p * rows + r]);
        for (int k = 0; k < d; ++k) O[r * d + k] = 0.0;
        if (m == ninf) {
            LSE[r] = ninf;
            continue;
        }
        double s = 0.0;
        for (int p = 0; p < n_parts; ++p) s += std::exp(LSE_parts[(int64_t)p * rows + r] - m);
        const double L = m + std::log(s);
        LSE[r] = L;
        for (int p = 0; p < n_parts; ++p) {
            const double lp = LSE_parts[(int64_t)p * rows + r];
            if (lp == ninf) continue;
            const double w = std::exp(lp - L);
            const double* op = O_parts + ((int64_t)p * rows + r) * d;
            for (int k = 0; k < d; ++k) O[r * d + k] += w * op[k];
        }
    }
}

// p, unclamped p_hat and (optionally clamped) p_hat of one row.
void orc_row_dists(const float* z, const float* q, int V, double T, double eta, int clamp,
                   double* p, double* phat_raw, double* phat) {
    row_dists(z, q, V, T, eta, clamp, p, phat_raw, phat);
}

void orc_residual_weights(const double* p, const double* phat, const float* q, int V, double* w) {
    residual_weights(p, phat, q, V, w);
}

int orc_sample_inverse_cdf(const double* w, int V, double u) {
    return sample_inverse_cdf(w, V, u, nullptr, nullptr);
}

// T^2 KL(q || softmax(z/T))  (Proposition 1's distillation loss).
double orc_kd_loss(const double* z, const double* q, int V, double T) {
    double m = -std::numeric_limits<double>::infinity();
    for (int k = 0; k < V; ++k) m = std::max(m, z[k] / T);
    double s = 0.0;
    for (int k = 0; k < V; ++k) s += std::exp(z[k] / T - m);
    const double log_s = std::log(s);
    double kl = 0.0;
    for (int k = 0; k < V; ++k) {
        if (q[k] <= 0.0) continue;
        const double log_p = z[k] / T - m - log_s;
        kl += q[k] * (std::log(q[k]) - log_p);
    }
    return T * T * kl;
}

// Proposition 1's closed form T (p - q), and the distilled logit
// z_hat = z - eta * dL/dz = z + eta T (q - p).
void orc_kd_grad(const double* z, const double* q, int V, double T, double* grad) {
    double m = -std::numeric_limits<double>::infinity();
    for (int k = 0; k < V; ++k) m = std::max(m, z[k] / T);
    double s = 0.0;
    for (int k = 0; k < V; ++k) s += std::exp(z[k] / T - m);
    for (int k = 0; k < V; ++k) grad[k] = T * (std::exp(z[k] / T - m) / s - q[k]);
}

void orc_distilled_logits(const double* z, const double* q, int V, double T, double eta,
                          double* z_hat) {
    std::vector<double> g(V);
    orc_kd_grad(z, q, V, T, g.data());
    for (int k = 0; k < V; ++k) z_hat[k] = z[k] - eta * g[k];
}

// The whole acceptance step.  diag [B,n_q,5] and sample_info [B,6] (row e,
// kind 0=bonus/1=residual/2=residual fell back to p, u, W, u*W, token) are
// optional.
void orc_accept(const float* z, const float* q, const int32_t* tokens, const int32_t* parent,
                const int32_t* n_nodes, int B, int n_q, int V, double T, double eta,
                uint64_t seed, int clamp, int32_t* n_acc, int32_t* next_tok, int32_t* path,
                double* diag, double* sample_info, int nthreads) {
    AcceptProblem A{z, q, tokens, parent, n_nodes, B, n_q, V, T, eta, seed, clamp};
    parallel_for(B, nthreads, [&](int64_t b) {
        accept_one(A, (int)b, n_acc, next_tok, path, diag, sample_info);
    });
}

// Brute-force sampling of the first emitted token with one draft (gamma = 1).
// Trial n: the draft token t ~ q_0 is drawn by inverse CDF from word 2 of
// Philox block {1, 0, 0, 0} under key seed + n (words 0 and 1 of that block
// are the method's r_1 and u_1); the step then accepts t or draws the next
// token from row 0.  hist[k] counts how often token k came out first.
void orc_first_token_hist(const float* z, const float* q, int V, double T, double eta, int clamp,
                          uint64_t seed, int64_t n_trials, int64_t* hist, int nthreads) {
    std::vector<double> p(V), raw(V), ph(V), w(V), qd(V);
    row_dists(z, q, V, T, eta, clamp, p.data(), raw.data(), ph.data());
    residual_weights(p.data(), ph.data(), q, V, w.data());
    double W = 0.0;
    for (int k = 0; k < V; ++k) W += w[k];
    if (!(W > 0.0)) w = p;
    for (int k = 0; k < V; ++k) qd[k] = q[k];
    const int nt = std::max(1, nthreads);
    std::vector<std::vector<int64_t>> local(nt, std::vector<int64_t>(V, 0));
    parallel_for(nt, nt, [&](int64_t w_id) {
        for (int64_t n = w_id; n < n_trials; n += nt) {
            const uint64_t s = seed + (uint64_t)n;
            uint32_t ctr[4] = {1u, 0u, 0u, 0u};
            uint32_t key[2] = {(uint32_t)(s & 0xffffffffu), (uint32_t)(s >> 32)};
            uint32_t out[4];
            philox4x32_10(ctr, key, out);
            const int t = sample_inverse_cdf(qd.data(), V, word_to_uniform(out[2]), nullptr, nullptr);
            const double r = word_to_uniform(out[0]);
            const double u = word_to_uniform(out[1]);
            const double ratio = q[t] == 0.0f ? std::numeric_limits<double>::infinity()
                                              : ph[t] / (double)q[t];
            int tok = t;
            if (!(r <= std::min(1.0, ratio))) tok = sample_inverse_cdf(w.data(), V, u, nullptr, nullptr);
            local[w_id][tok]++;
        }
    });
    for (int k = 0; k < V; ++k) {
        hist[k] = 0;
        for (int w_id = 0; w_id < nt; ++w_id) hist[k] += local[w_id][k];
    }
}

}  // extern "C"
