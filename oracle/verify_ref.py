"""Float64 CPU oracle for the speculative-decoding verify step (gated NoPE MLA).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg import this module.  It shares no code with the
CUDA library and imports nothing from it.

What it computes, written as the plain definitions (no blocking, no fusion):

* Attention (``ref_verify_attention``).  Each request feeds one verify group
  of 1 target token plus k drafted tokens ("M* PR #257 - Kimi K3 support with
  DSpark speculative decoding", section "Speculative decoding").  Attention is
  absorbed NoPE MLA ("... gated NoPE MLA runs on FlashInfer with absorbed
  projections", same PR, section "Model"): the query of every head lives in
  the 512-wide latent space, and the cached latent row c_j is both key and
  value.  Token t of request r attends to KV positions j < kv_bounds[t]
  (the per-token attention bound local_len(pos + 1) of "TensorRT-LLM PR #18166
  - Kimi K3: DSpark speculative decoding under Helix CP", Summary and first
  commit).  Scores s_j = scale * <q, c_j>; lse = log sum_j exp(s_j) (natural
  log); o = sum_j exp(s_j - lse) c_j.  A bound of 0 gives the (-inf, 0)
  identity: lse = -inf and o = 0 (same PR, first commit "stats epilogue emits
  the (-inf, 0) identity per token").
* Gate.  out = sigmoid(gate) * o elementwise over the 512 latent columns
  ("gated NoPE MLA"; the pages give no gate shape, this reading is a
  [T, H, 512] elementwise sigmoid gate applied to the normalised output).
  PARITY UNPINNED for the gate's shape and placement: the pages do not fix
  them; the pins below only fix sigmoid(g) * o for the reading taken.
* Head-wise gate.  A gate of shape [T, H] (one value per token and head)
  scales the whole 512-wide latent row: out = sigmoid(gate[t, h]) * o[t, h]
  ("next" variant of the Kimi K3 helix configuration in "TensorRT-LLM PR
  #18166", which runs H = 96; a head-wise gate is the form that commutes
  with the per-head value up-projection W_UV).
* Value up-projection (``ref_wuv_project``): the absorbed latent output of
  head h is mapped to the head's value space by W_UV[h] (v_dim x 512):
  v[t, h] = W_UV[h] @ out[t, h] ("LSE combine + W_UV" after the context-
  parallel merge, vLLM page "kimi_k3/nvidia/specialized_decode/drafter/
  model"; absorbed MLA keeps W_UV out of the attention).
* fp8 latent KV (``e4m3_bits_to_f64``): a page pool of OCP FP8 E4M3 codes
  (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; subnormals;
  S.1111.111 is NaN, no infinities) with one scale for the whole pool; the
  cached latent row is code value x kv_scale.  The attention over it is the
  plain definition applied to those dequantised rows (the model card
  "RedHatAI/Kimi-K3-speculator.dspark", section "Deployment", serves the
  target with an fp8 KV cache; "TensorRT-LLM PR #18166" keeps fp8 KV out of
  its verify kernel, so this is the "next" variant).
* Split-KV partials and their merge (``ref_attention_partials``,
  ``ref_lse_combine``): each KV range gives (o_s, lse_s) by the same formula;
  lse = log sum_s exp(lse_s), o = sum_s exp(lse_s - lse) o_s, and an all
  -inf set gives (-inf, 0) rather than NaN (the CP-merge weighting of
  "TensorRT-LLM PR #18166", second and third commits: corr = 0 for a
  zero-bound row, never 0 * NaN).
* Paged KV append (``ref_kv_append``): the latent rows of the k+1 verify
  tokens are written into the page pool at their positions before the
  attention reads them: position pos of request r lands in page
  block_table[r][pos // page_size], slot pos % page_size; a position of -1
  writes nothing (the per-token KV write slot of "TensorRT-LLM PR #18166",
  first commit message, "-1 = not owned"; one GPU owns every position).
* Greedy verify (``ref_greedy_verify``): a_t = argmax_v logits[t, v] (lowest
  index on ties); accepted n_r = largest m <= k with d_j = a_{j-1} for all
  j <= m; next token a_{n_r}; the KV trims the rejected tail:
  kv_lens_out = kv_lens_in - (k - n_r) ("M* PR #257", section "Speculative
  decoding": verification is greedy, the KV trims rejected tails).

Inputs are numpy arrays as built by ``workloads.make_inputs``: bf16 values are
raw uint16 bit patterns and are widened to float64 exactly.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def e4m3_bits_to_f64(codes: np.ndarray) -> np.ndarray:
    """Exact value of FP8 E4M3 codes (uint8), from the format's definition."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = sign * (1.0 + m / 8.0) * np.power(2.0, e - 7)
    sub = sign * (m / 8.0) * 2.0 ** -6
    v = np.where(e == 0, sub, normal)
    return np.where((c & 0x7F) == 0x7F, np.nan, v)


def gather_latent_rows(kv_pages: np.ndarray, block_row: np.ndarray, n: int) -> np.ndarray:
    """Rows 0..n-1 of one request's latent sequence: position j lives in page
    block_row[j // page_size] at slot j % page_size (paged KV, block table)."""
    page_size = kv_pages.shape[1]
    if n == 0:
        return np.zeros((0, kv_pages.shape[2]), dtype=kv_pages.dtype)
    j = np.arange(n)
    pages = np.asarray(block_row)[j // page_size]
    if np.any(pages < 0) or np.any(pages >= kv_pages.shape[0]):
        raise ValueError("block table entry outside the page pool")
    return kv_pages[pages, j % page_size]


def sigmoid(x: np.ndarray) -> np.ndarray:
    """Logistic function 1 / (1 + exp(-x)), evaluated without overflow."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    pos = x >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-x[pos]))
    ex = np.exp(x[~pos])
    out[~pos] = ex / (1.0 + ex)
    return out


def _softmax_stats(s: np.ndarray, rows: np.ndarray):
    """(lse, o) of scores s[h, j] over latent rows[j]; empty -> (-inf, 0)."""
    H = s.shape[0]
    D = rows.shape[1]
    if s.shape[1] == 0:
        return np.full(H, -np.inf), np.zeros((H, D))
    m = s.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(s - m).sum(axis=1))
    p = np.exp(s - lse[:, None])
    return lse, p @ rows


def ref_verify_attention(q, kv_pages, block_table, kv_bounds, gate, q_per_req, softmax_scale):
    """Gated, absorbed NoPE MLA decode attention with per-token bounds.

    q: [T, H, D], gate: [T, H, D] (elementwise) or [T, H] (head-wise), float64
    or bf16 bits; kv_pages: [P, page, D]; block_table: [R, max_pages];
    kv_bounds: [T].  Returns (out [T, H, D], lse [T, H]) in float64; out is
    gated, lse is of the ungated scaled scores.
    """
    q = _as_f64(q)
    g = _as_f64(gate)
    T, H, D = q.shape
    out = np.zeros((T, H, D))
    lse = np.full((T, H), -np.inf)
    R = (T + q_per_req - 1) // q_per_req if q_per_req > 0 else 0
    for r in range(R):
        toks = range(r * q_per_req, min(T, (r + 1) * q_per_req))
        # one gather per request; each token then sees a prefix of it
        rows_all = _as_f64(gather_latent_rows(kv_pages, block_table[r],
                                              max(int(kv_bounds[t]) for t in toks)))
        for t in toks:
            rows = rows_all[:int(kv_bounds[t])]
            s = softmax_scale * (q[t] @ rows.T)
            lse[t], o = _softmax_stats(s, rows)
            out[t] = gate_factor(g[t]) * o
    return out, lse


def gate_factor(g_t: np.ndarray) -> np.ndarray:
    """sigmoid of one token's gate, shaped to multiply its [H, D] output: a
    head-wise gate [H] becomes a column [H, 1]."""
    sg = sigmoid(g_t)
    return sg[:, None] if sg.ndim == 1 else sg


def ref_wuv_project(out_latent, w_uv) -> np.ndarray:
    """Per-head value up-projection v[t, h, :] = W_UV[h] @ out[t, h, :].

    out_latent [T, H, D] (float64 or bf16 bits), w_uv [H, v_dim, D] (float64 or
    bf16 bits).  Returns [T, H, v_dim] float64."""
    x = _as_f64(out_latent)
    w = _as_f64(w_uv)
    T, H, D = x.shape
    v = np.zeros((T, H, w.shape[1]))
    for h in range(H):
        v[:, h, :] = x[:, h, :] @ w[h].T
    return v


def ref_attention_partials(q, kv_pages, block_table, kv_bounds, q_per_req, softmax_scale, edges):
    """Split-KV partials: split s of request r covers positions
    [edges[r][s], edges[r][s+1]) intersected with each token's bound.

    Returns part_o [S, T, H, D] (normalised within the split) and
    part_lse [S, T, H]; an empty range gives (lse=-inf, o=0)."""
    q = _as_f64(q)
    T, H, D = q.shape
    S = len(edges[0]) - 1 if len(edges) else 0
    part_o = np.zeros((S, T, H, D))
    part_lse = np.full((S, T, H), -np.inf)
    for t in range(T):
        r = t // q_per_req
        b = int(kv_bounds[t])
        rows = _as_f64(gather_latent_rows(kv_pages, block_table[r], b))
        for s_i in range(S):
            lo = int(edges[r][s_i])
            hi = min(int(edges[r][s_i + 1]), b)
            seg = rows[lo:hi] if hi > lo else rows[:0]
            sc = softmax_scale * (q[t] @ seg.T)
            part_lse[s_i, t], part_o[s_i, t] = _softmax_stats(sc, seg)
    return part_o, part_lse


def ref_lse_combine(part_o, part_lse, gate=None):
    """Merge split partials by their LSE; optional sigmoid gate epilogue.

    lse = log sum_s exp(lse_s); o = sum_s exp(lse_s - lse) o_s; rows whose
    partials are all -inf give (lse=-inf, o=0)."""
    part_o = np.asarray(part_o, dtype=np.float64)
    part_lse = np.asarray(part_lse, dtype=np.float64)
    m = part_lse.max(axis=0)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    w_raw = np.exp(part_lse - m_safe[None])
    z = w_raw.sum(axis=0)
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, z)))
    w = np.where(empty[None], 0.0, w_raw / np.where(empty, 1.0, z)[None])
    o = (w[..., None] * part_o).sum(axis=0)
    if gate is not None:
        g = sigmoid(_as_f64(gate))
        o = (g[..., None] if g.ndim == o.ndim - 1 else g) * o
    return o, lse


def ref_greedy_verify(logits, draft_tokens, kv_lens_in, k):
    """Greedy verification and KV trim.

    logits [T, V] (T = R (k+1)), draft_tokens [R, k], kv_lens_in [R].
    Returns (argmax [T], accepted [R], next_tokens [R], kv_lens_out [R])."""
    x = np.asarray(logits, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("logits must be finite")
    R = int(np.asarray(kv_lens_in).shape[0])
    T = x.shape[0]
    assert T == R * (k + 1)
    a = np.argmax(x, axis=1).astype(np.int64) if x.shape[1] > 0 else np.zeros(T, np.int64)
    accepted = np.zeros(R, dtype=np.int64)
    nxt = np.zeros(R, dtype=np.int64)
    kv_out = np.zeros(R, dtype=np.int64)
    for r in range(R):
        base = r * (k + 1)
        n = 0
        while n < k and int(draft_tokens[r][n]) == int(a[base + n]):
            n += 1
        accepted[r] = n
        nxt[r] = a[base + n]
        kv_out[r] = int(kv_lens_in[r]) - (k - n)
    return a, accepted, nxt, kv_out


def ref_kv_append(kv_pages, block_table, positions, kv_new, q_per_req):
    """Return a copy of the page pool with token t's latent row kv_new[t]
    stored at its position (request r = t // q_per_req); -1 skips the token."""
    pool = np.array(kv_pages, copy=True)
    page_size = pool.shape[1]
    for t, pos in enumerate(np.asarray(positions)):
        pos = int(pos)
        if pos < 0:
            continue
        r = t // q_per_req
        page = int(block_table[r][pos // page_size])
        if page < 0 or page >= pool.shape[0]:
            raise ValueError("block table entry outside the page pool")
        pool[page, pos % page_size] = kv_new[t]
    return pool


def ref_verify_step(inp: dict) -> dict:
    """The whole hot path on one batch from ``workloads.make_inputs``."""
    out, lse = ref_verify_attention(inp["q_bits"], inp["kv_bits"], inp["block_table"],
                                    inp["kv_bounds"], inp["gate_bits"], inp["k"] + 1,
                                    inp["softmax_scale"])
    a, n, nxt, kv_out = ref_greedy_verify(inp["logits"], inp["draft_tokens"],
                                          inp["kv_lens_in"], inp["k"])
    return dict(out=out, lse=lse, argmax=a, accepted=n, next_tokens=nxt, kv_lens_out=kv_out)


def _as_f64(x) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_bits_to_f64(x)
    return x.astype(np.float64, copy=False)
