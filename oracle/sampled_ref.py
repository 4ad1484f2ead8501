"""Float64 CPU oracle for sampled (rejection-sampling) speculative verification.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg import this module.  It shares no code with the
CUDA library and imports nothing from it.

"M* PR #257 - Kimi K3 support with DSpark speculative decoding", section
"Speculative decoding", says verification is greedy or sampled, the sampled
form being FlashInfer's chain sampling; the model card
"RedHatAI/Kimi-K3-speculator.dspark", section "Deployment", serves the draft
with probabilistic draft sampling (and names vLLM's block rejection method,
which is not modelled here).  The pages print no algorithm, so this is the
plain token-wise chain rejection sampling of the published speculative
sampling method (Leviathan, Kalman, Matias 2023; Chen et al. 2023), on one
verify group of 1 target + k drafted tokens per request:

* target distribution of verify token t: p_t = softmax(logits[t] / temperature);
* draft j (0-based) of request r was drawn from q_{r,j} = draft_probs[r][j];
  it is accepted iff u_{r,j} * q_{r,j}(d) < p_t(d), t = r (k+1) + j, i.e.
  with probability min(1, p/q) for a uniform u in [0, 1);
* at the first rejected j the next token is drawn from the residual
  w = max(0, p_t - q_{r,j}) (normalised); if every draft is accepted it is
  drawn from p of the last verify token (the bonus token); a residual that is
  zero everywhere (p = q) falls back to p_t;
* a draw from weights w with uniform u is the inverse CDF: the smallest v
  with sum_{i <= v} w_i > u * sum_i w_i;
* accepted n_r counts the accepted drafts; the KV keeps the target token and
  the accepted drafts: kv_lens_out = kv_lens_in - (k - n_r), as in greedy
  verification ("the KV trims rejected tails").

The random numbers are inputs: uniforms[r][0..k-1] decide the acceptances,
uniforms[r][k] draws the next token.
"""
from __future__ import annotations

import numpy as np


def target_probs(logits_row, temperature: float) -> np.ndarray:
    """softmax(x / temperature) in float64 (max-shifted)."""
    z = np.asarray(logits_row, dtype=np.float64) / float(temperature)
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


def inverse_cdf(w: np.ndarray, u: float) -> int:
    """Smallest v with sum_{i <= v} w_i > u * sum(w); w >= 0, sum(w) > 0."""
    c = np.cumsum(np.asarray(w, dtype=np.float64))
    v = int(np.searchsorted(c, float(u) * c[-1], side="right"))
    if v >= len(c):  # u * W rounded up to W: the last index with weight
        v = int(np.nonzero(np.asarray(w) > 0)[0][-1])
    return v


def ref_sampled_verify(logits, draft_tokens, draft_probs, uniforms, kv_lens_in, k: int,
                       temperature: float, detail: bool = False):
    """Sampled verification of R verify groups.

    logits [T, V] (T = R (k+1)), draft_tokens [R, k], draft_probs [R, k, V]
    (each row a distribution), uniforms [R, k+1] in [0, 1), kv_lens_in [R].
    Returns (accepted [R], next_tokens [R], kv_lens_out [R]); with detail=True
    also a list of per-request dicts holding the margins of every decision
    taken (relative gap of the acceptance test, CDF gap of the draw in units
    of the total weight) and the weights the next token was drawn from."""
    x = np.asarray(logits, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("logits must be finite")
    if not (temperature > 0 and np.isfinite(temperature)):
        raise ValueError("temperature must be positive and finite")
    R = int(np.asarray(kv_lens_in).shape[0])
    assert x.shape[0] == R * (k + 1)
    qd = np.asarray(draft_probs, dtype=np.float64)
    u = np.asarray(uniforms, dtype=np.float64)
    accepted = np.zeros(R, dtype=np.int64)
    nxt = np.zeros(R, dtype=np.int64)
    kv_out = np.zeros(R, dtype=np.int64)
    info = []
    for r in range(R):
        base = r * (k + 1)
        n = k
        w = None
        gaps = []
        for j in range(k):
            p = target_probs(x[base + j], temperature)
            d = int(draft_tokens[r][j])
            lhs, rhs = u[r, j] * qd[r, j, d], p[d]
            gaps.append(abs(rhs - lhs) / max(rhs, lhs, 1e-300))
            if lhs < rhs:
                continue
            n = j
            w = np.maximum(p - qd[r, j], 0.0)
            if not np.any(w > 0):
                w = p
            break
        if w is None:
            w = target_probs(x[base + k], temperature)
        v = inverse_cdf(w, u[r, k])
        accepted[r] = n
        nxt[r] = v
        kv_out[r] = int(kv_lens_in[r]) - (k - n)
        if detail:
            c = np.cumsum(w)
            tgt = u[r, k] * c[-1]
            lo = c[v - 1] if v > 0 else 0.0
            info.append(dict(accept_gaps=gaps, draw_gap=min(tgt - lo, c[v] - tgt) / c[-1],
                             weights=w, target=tgt, cdf=c))
    if detail:
        return accepted, nxt, kv_out, info
    return accepted, nxt, kv_out
