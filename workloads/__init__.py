"""Seeded synthetic inputs for the speculative-decoding verify step.

This module builds the inputs that both the CUDA path and the float64 oracle
read: the bf16 query latents, the paged bf16 latent KV pool with its block
table, the per-token causal bounds, the gate, the fp32 target logits and the
draft tokens.  It holds none of the verify step's arithmetic (no attention,
no softmax, no argmax): every value is drawn or placed by construction.

Workloads (sizes as named by the verify-step configurations):

* ``c0`` tiny verify: 2 requests, k=3, H=8, KV lengths 64 and 100,
  logits vocab 1024 ~ N(0, 1), draft match p=0.5.
* ``c1`` C=1 verify: 1 request, k=7, H=64, context 1536, logits
  [8, 163840] ~ N(0, 2), draft match p=0.6.
* ``c2`` C=32 verify: 32 requests, k=4, H=64, contexts U[1024, 1536],
  shuffled block tables, logits [160, 163840], p=0.6.
* ``c3`` C=64 plain decode: 64 requests, k=0, H=64, contexts U[1024, 1536].
* ``c4`` long-context verify: 16 requests, k=7, H=64, contexts U[8192, 32768];
  half the requests get ``L mod 64`` in ``[1, k]`` so that the verify group
  straddles a page; 10% of query tokens get bound 0.

Recipe (seed 0 unless given):

1. ``kv_lens_in`` (fixed, or uniform integers in the closed range), then the
   straddle adjustment, then the zero-bound token choice, then the page
   permutation.
2. ``q``, the KV pool, ``gate``: float32 N(0, 1) draws rounded to bf16
   (round to nearest even) and kept as raw uint16 bit patterns.
3. ``logits``: float32 N(0, sd) draws clipped to +-5.5 sd; for each token a
   target id drawn uniformly is then set to 6 sd, so the row's maximum sits at
   that planted id by construction.
4. Drafts: ``d_j`` (j = 1..k) equals the planted target of token j-1 with
   probability p, otherwise a uniform id different from it.

Causal bounds follow "token at position pos sees KV positions < pos + 1":
the k+1 verify tokens of request r sit at positions ``L_r - k - 1 .. L_r - 1``
(``L_r`` = kv_lens_in[r] already counts them), so token t sees
``b = L_r - k + t`` rows.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np

PAGE_SIZE = 64
LATENT_DIM = 512


@dataclass(frozen=True)
class VerifyConfig:
    name: str
    R: int                      # requests (verify groups)
    k: int                      # drafted tokens per group; group = k + 1 tokens
    H: int                      # query heads
    vocab: int
    logit_sd: float
    draft_p: float
    kv_lens: tuple | None = None        # fixed per-request lengths
    kv_len_range: tuple | None = None   # inclusive uniform range
    shuffled: bool = False
    straddle_half: bool = False
    zero_bound_frac: float = 0.0
    softmax_scale: float = 1.0 / math.sqrt(128.0)
    D: int = LATENT_DIM
    page_size: int = PAGE_SIZE
    description: str = field(default="", compare=False)

    @property
    def q_per_req(self) -> int:
        return self.k + 1

    @property
    def T(self) -> int:
        return self.R * (self.k + 1)


CONFIGS = {
    "c0": VerifyConfig("c0", R=2, k=3, H=8, vocab=1024, logit_sd=1.0, draft_p=0.5,
                       kv_lens=(64, 100),
                       description="tiny verify: 2 requests, k=3, H=8, KV 64/100"),
    "c1": VerifyConfig("c1", R=1, k=7, H=64, vocab=163840, logit_sd=2.0, draft_p=0.6,
                       kv_lens=(1536,),
                       description="C=1 decode verify: 1 request, k=7, H=64, context 1536"),
    "c2": VerifyConfig("c2", R=32, k=4, H=64, vocab=163840, logit_sd=2.0, draft_p=0.6,
                       kv_len_range=(1024, 1536), shuffled=True,
                       description="C=32 verify: 32 requests, k=4, H=64, contexts U[1024,1536]"),
    "c3": VerifyConfig("c3", R=64, k=0, H=64, vocab=163840, logit_sd=2.0, draft_p=0.6,
                       kv_len_range=(1024, 1536), shuffled=True,
                       description="C=64 plain decode: 64 requests, k=0, H=64, contexts U[1024,1536]"),
    "c4": VerifyConfig("c4", R=16, k=7, H=64, vocab=163840, logit_sd=2.0, draft_p=0.6,
                       kv_len_range=(8192, 32768), shuffled=True, straddle_half=True,
                       zero_bound_frac=0.10,
                       description="long-context split-KV verify: 16 requests, k=7, H=64, "
                                   "contexts U[8192,32768], straddling groups, 10% bound-0 tokens"),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def _normal_bf16(rng: np.random.Generator, shape, chunk_rows: int = 4096) -> np.ndarray:
    """N(0, 1) float32 draws rounded to bf16, generated row-chunk by row-chunk.

    Drawing in chunks from one generator yields the same stream as one big draw,
    and keeps the float32 temporary small for the large KV pools."""
    shape = tuple(shape)
    out = np.empty(shape, dtype=np.uint16)
    flat = out.reshape(shape[0], -1)
    inner = flat.shape[1]
    for s in range(0, shape[0], chunk_rows):
        e = min(shape[0], s + chunk_rows)
        flat[s:e] = f32_to_bf16_bits(rng.standard_normal((e - s, inner), dtype=np.float32))
    return out


def causal_bounds(kv_lens_in: np.ndarray, k: int) -> np.ndarray:
    """Per-token bound b = L - k + t for token t = 0..k of each request."""
    t = np.arange(k + 1, dtype=np.int64)
    return (kv_lens_in.astype(np.int64)[:, None] - k + t[None, :]).reshape(-1).astype(np.int32)


def make_inputs(cfg: VerifyConfig | str, seed: int = 0) -> dict:
    """Build one seeded verify-step batch (numpy arrays, host memory)."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    rng = np.random.default_rng(seed)
    R, k, H, D, ps = cfg.R, cfg.k, cfg.H, cfg.D, cfg.page_size
    T = R * (k + 1)

    # 1. structure
    if cfg.kv_lens is not None:
        kv_lens = np.asarray(cfg.kv_lens, dtype=np.int64)
        assert kv_lens.shape == (R,)
    else:
        lo, hi = cfg.kv_len_range
        kv_lens = rng.integers(lo, hi + 1, size=R, dtype=np.int64)
    if cfg.straddle_half and k > 0:
        chosen = rng.choice(R, size=R // 2, replace=False)
        rem = rng.integers(1, k + 1, size=chosen.size)
        for r, x in zip(chosen, rem):
            L = (int(kv_lens[r]) // ps) * ps + int(x)
            if cfg.kv_len_range is not None and L > cfg.kv_len_range[1]:
                L -= ps
            kv_lens[r] = L
    kv_lens = kv_lens.astype(np.int32)
    kv_bounds = causal_bounds(kv_lens, k)
    if cfg.zero_bound_frac > 0:
        nz = int(round(cfg.zero_bound_frac * T))
        zero_tokens = np.sort(rng.choice(T, size=nz, replace=False))
        kv_bounds[zero_tokens] = 0
    else:
        zero_tokens = np.zeros(0, dtype=np.int64)

    pages_per_req = (kv_lens.astype(np.int64) + ps - 1) // ps
    num_pages = int(pages_per_req.sum())
    max_pages = int(pages_per_req.max()) if R > 0 else 0
    if cfg.shuffled:
        perm = rng.permutation(num_pages)
    else:
        perm = np.arange(num_pages)
    block_table = np.full((R, max(max_pages, 1)), -1, dtype=np.int32)
    off = 0
    for r in range(R):
        n = int(pages_per_req[r])
        block_table[r, :n] = perm[off:off + n]
        off += n

    # 2. values
    q = _normal_bf16(rng, (T, H, D))
    kv = _normal_bf16(rng, (num_pages, ps, D), chunk_rows=64)
    gate = _normal_bf16(rng, (T, H, D))

    # 3. logits with a planted per-row maximum
    V = cfg.vocab
    sd = cfg.logit_sd
    logits = np.empty((T, V), dtype=np.float32)
    for t in range(T):
        logits[t] = np.clip(rng.standard_normal(V, dtype=np.float32) * np.float32(sd),
                            -5.5 * sd, 5.5 * sd)
    planted = rng.integers(0, V, size=T).astype(np.int32)
    logits[np.arange(T), planted] = np.float32(6.0 * sd)

    # 4. drafts: d_j copies the planted target of token j-1 with probability p
    coins = rng.random((R, k))
    others = rng.integers(0, V - 1, size=(R, k))
    draft = np.empty((R, k), dtype=np.int32)
    for r in range(R):
        for j in range(1, k + 1):
            target = int(planted[r * (k + 1) + j - 1])
            if coins[r, j - 1] < cfg.draft_p:
                draft[r, j - 1] = target
            else:
                u = int(others[r, j - 1])
                draft[r, j - 1] = u + (1 if u >= target else 0)

    return dict(
        cfg=cfg, seed=seed, R=R, k=k, H=H, D=D, T=T, page_size=ps,
        num_pages=num_pages, max_pages=block_table.shape[1],
        softmax_scale=float(cfg.softmax_scale),
        kv_lens_in=kv_lens, kv_bounds=kv_bounds, zero_bound_tokens=zero_tokens.astype(np.int32),
        block_table=block_table, q_bits=q, kv_bits=kv, gate_bits=gate,
        logits=logits, planted_argmax=planted, draft_tokens=draft,
    )


def make_sampled_inputs(cfg: VerifyConfig | str, seed: int = 0, temperature: float = 1.0,
                        draft_mix: tuple[float, float] = (0.05, 0.95)) -> dict:
    """Inputs of sampled verification for one batch (numpy, host memory).

    Its own random stream (seed, 2), so it does not disturb ``make_inputs``.
    Target logits follow the same recipe as ``make_inputs`` (N(0, sd) clipped
    to +-5.5 sd, one planted id per row at 6 sd).  Draft position j of request
    r has the distribution q = (1 - a_r) * onehot(planted id of token j) +
    a_r * E / sum(E), E ~ Exp(1) iid over the vocabulary, a_r ~ U(draft_mix),
    stored as float32; the draft token is drawn from q (numpy's categorical
    draw).  Uniforms [R][k+1] ~ U[0, 1)."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    rng = np.random.default_rng([seed, 2])
    R, k, V, sd = cfg.R, cfg.k, cfg.vocab, cfg.logit_sd
    T = R * (k + 1)
    if cfg.kv_lens is not None:
        kv_lens = np.asarray(cfg.kv_lens, dtype=np.int32)
    else:
        lo, hi = cfg.kv_len_range
        kv_lens = rng.integers(lo, hi + 1, size=R).astype(np.int32)
    logits = np.empty((T, V), dtype=np.float32)
    for t in range(T):
        logits[t] = np.clip(rng.standard_normal(V, dtype=np.float32) * np.float32(sd),
                            -5.5 * sd, 5.5 * sd)
    planted = rng.integers(0, V, size=T).astype(np.int32)
    logits[np.arange(T), planted] = np.float32(6.0 * sd)
    mix = rng.uniform(draft_mix[0], draft_mix[1], size=R)
    draft_probs = np.empty((R, k, V), dtype=np.float32)
    drafts = np.empty((R, k), dtype=np.int32)
    for r in range(R):
        for j in range(k):
            e = rng.exponential(1.0, size=V)
            q = mix[r] * e / e.sum()
            q[planted[r * (k + 1) + j]] += 1.0 - mix[r]
            draft_probs[r, j] = q.astype(np.float32)
            drafts[r, j] = rng.choice(V, p=q / q.sum())
    uniforms = rng.random((R, k + 1)).astype(np.float32)
    return dict(cfg=cfg, seed=seed, R=R, k=k, T=T, V=V, temperature=float(temperature),
                kv_lens_in=kv_lens, logits=logits, planted_argmax=planted,
                draft_probs=draft_probs, draft_tokens=drafts, uniforms=uniforms)


def fp8_kv_pool(inp: dict, amax_target: float = 448.0) -> tuple[np.ndarray, float]:
    """An FP8 E4M3 page pool for the batch of ``make_inputs``: the bf16 latent
    rows scaled by 1 / kv_scale (kv_scale = max |row value| / 448, so the pool
    spans the format's range) and rounded to the nearest E4M3 code (torch's
    float8_e4m3fn conversion).  Returns (codes uint8 [P][64][512], kv_scale)."""
    import torch
    kv = torch.from_numpy(np.ascontiguousarray(inp["kv_bits"]).view(np.int16)).view(torch.bfloat16).float()
    amax = float(kv.abs().max())
    kv_scale = amax / amax_target if amax > 0 else 1.0
    codes = (kv / kv_scale).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return codes, float(kv_scale)


def small_config(base: str | VerifyConfig = "c0", **overrides) -> VerifyConfig:
    """A variant of a named configuration (edge cases, test sweeps)."""
    if isinstance(base, str):
        base = CONFIGS[base]
    return replace(base, **overrides)
