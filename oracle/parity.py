"""TEST INFRASTRUCTURE: counting the near-boundary cases of an acceptance
comparison (CUDA path vs this oracle) without failing on them.

Used by ``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg to report
how many decisions the stated exemption bands covered; the GPU test suite
asserts the same bands in tests/_parity.py.  Decisions are those of the ratio
test of "RAPID: Long-Context Inference with Retrieval-Augmented Speculative
Decoding" (blog summary), section 2.1, with the retrieval-augmented target and
its tail rule of section 2.4.  A decision may differ only where the uniform
sits within 1e-5 of its boundary: |r - ratio| < 1e-5, p_hat(t) within 1e-5
(relative) of the 0.1 max p_hat tail threshold, or, for the drawn token,
|u W - C_k| < 1e-5 W at an inverse-CDF boundary.
"""
import numpy as np

from . import residual_weights, row_dists

BAND = 1e-5


def accept_exemptions(z, q, tokens, parent, T, eta, clamp, gpu, ref):
    """Counts for one call: z, q [B, n_q, V]; tokens, parent [B, n_q] (parent
    None for a chain); gpu / ref: dicts of numpy arrays n_accepted, next_token,
    path, diag (ref from oracle.accept, with its 'sample' record).

    Returns dict(sequences, compared, ratio_exempt, clamp_exempt, cdf_exempt,
    mismatched): a sequence with a decision inside a band is counted and not
    compared further; 'mismatched' counts differences outside every band."""
    B, n_q, _ = z.shape
    out = dict(sequences=0, compared=0, ratio_exempt=0, clamp_exempt=0, cdf_exempt=0,
               mismatched=0)
    for b in range(B):
        out["sequences"] += 1
        parents = [-1] + ([int(x) for x in parent[b][1:]] if parent is not None
                          else list(range(n_q - 1)))
        kind_ex = None
        for i in range(1, n_q):
            dg, dr = gpu["diag"][b, i], ref["diag"][b, i]
            if (dg[4] <= min(1.0, dg[3])) == (dr[4] <= min(1.0, dr[3])):
                continue
            near_clamp = False
            if clamp:
                _, raw, _ = row_dists(z[b, parents[i]], q[b, parents[i]], T, eta, True)
                thr = 0.1 * raw.max()
                near_clamp = abs(raw[int(tokens[b, i])] - thr) <= BAND * thr
            if near_clamp:
                kind_ex = "clamp_exempt"
            elif abs(dr[4] - dr[3]) < BAND:
                kind_ex = kind_ex or "ratio_exempt"
            else:
                kind_ex = "mismatched"
                break
        if kind_ex is not None:
            out[kind_ex] += 1
            continue
        out["compared"] += 1
        if gpu["n_accepted"][b] != ref["n_accepted"][b] or (
                gpu.get("path") is not None and not np.array_equal(gpu["path"][b], ref["path"][b])):
            out["mismatched"] += 1
            continue
        tg, to = int(gpu["next_token"][b]), int(ref["next_token"][b])
        if tg == to:
            continue
        e, kind, _, W, target = ref["sample"][b][:5]
        p, _, ph = row_dists(z[b, int(e)], q[b, int(e)], T, eta, clamp)
        w = residual_weights(p, ph, q[b, int(e)]) if int(kind) == 1 else p
        C = np.cumsum(w)
        gaps = np.abs(C[min(tg, to):max(tg, to)] - target)
        out["cdf_exempt" if (gaps < BAND * W).all() else "mismatched"] += 1
    return out
