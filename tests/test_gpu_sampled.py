"""GPU parity of sampled (rejection-sampling) verification against the float64
oracle, called through the C ABI.

The kernels take their decisions in fp32, the oracle in float64.  A decision
whose oracle margin is wider than the fp32 error bound must come out the same;
one inside it may go either way, and the test then checks that the GPU's
choice is one of the valid ones.  An ambiguous acceptance does not exempt its
request: the oracle is run again on that request with the decision forced to
the GPU's choice (uniform 0 forces an acceptance, +inf a rejection), so every
other decision, the trim and the draw that follow are still compared.
* acceptance: relative gap |u q - p| / max(u q, p) below ACCEPT_TOL (fp32
  products and the ex2-based softmax carry ~1e-6 relative error);
* draw: the GPU's id v must have positive weight and a CDF step
  [c_{v-1}, c_v] that holds u W within DRAW_TOL W (fp32 sums of up to 2^17
  non-negative terms in 1024-element tiles: well below 1e-5 W).
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import CONFIGS, make_inputs, make_sampled_inputs, small_config

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
ACCEPT_TOL = 1e-4
DRAW_TOL = 2e-5


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verify_mla_gb300 as m
    m.load_library()
    return m


def _dev(inp):
    f = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).to(DEV)  # noqa: E731
    return (f(inp["logits"], np.float32), f(inp["draft_tokens"], np.int32), f(inp["draft_probs"], np.float32),
            f(inp["uniforms"], np.float32), f(inp["kv_lens_in"], np.int32))


def run_gpu(sv, inp, temperature=None):
    lg, dt, dp, un, kv = _dev(inp)
    temp = inp["temperature"] if temperature is None else temperature
    res = sv.spec_verify_sampled(lg, dt, dp, un, kv, inp["k"], temperature=temp)
    torch.cuda.synchronize()
    return [r.cpu().numpy().astype(np.int64) for r in res]


def _oracle_following_gpu(inp, r, ga_r, temp):
    """The oracle on request r alone, with every acceptance test whose margin
    is inside ACCEPT_TOL forced to the decision the GPU took there (the GPU
    accepted drafts 0..ga_r-1 and rejected draft ga_r).  Returns (accepted,
    next token, detail, number of forced decisions)."""
    k = inp["k"]
    rows = slice(r * (k + 1), (r + 1) * (k + 1))
    u = np.asarray(inp["uniforms"][r:r + 1], dtype=np.float64).copy()
    forced = set()
    while True:
        a, nxt, _, info = oracle.ref_sampled_verify(inp["logits"][rows], inp["draft_tokens"][r:r + 1],
                                                    inp["draft_probs"][r:r + 1], u, inp["kv_lens_in"][r:r + 1],
                                                    k, temp, detail=True)
        amb = [j for j, g in enumerate(info[0]["accept_gaps"]) if g < ACCEPT_TOL and j not in forced]
        if not amb:
            return int(a[0]), int(nxt[0]), info[0], len(forced)
        j = amb[0]
        assert j <= ga_r, (f"request {r}: the GPU rejected draft {ga_r} although the oracle's decision "
                           "there is clear")
        u[0, j] = 0.0 if j < ga_r else np.inf
        forced.add(j)


def check_sampled(inp, got, temperature=None, max_ambiguous_frac=0.1):
    temp = inp["temperature"] if temperature is None else temperature
    k = inp["k"]
    a, nxt, kv, info = oracle.ref_sampled_verify(inp["logits"], inp["draft_tokens"], inp["draft_probs"],
                                                 inp["uniforms"], inp["kv_lens_in"], k, temp, detail=True)
    ga, gn, gkv = got
    R = len(a)
    assert np.all((ga >= 0) & (ga <= k))
    assert np.array_equal(gkv, np.asarray(inp["kv_lens_in"]) - (k - ga)), "trim must follow accepted"
    ambiguous = 0
    draws_checked = 0
    for r in range(R):
        gaps = info[r]["accept_gaps"]
        a_r, n_r, info_r = a[r], nxt[r], info[r]
        if gaps and min(gaps) < ACCEPT_TOL:
            ambiguous += 1
            a_r, n_r, info_r, n_forced = _oracle_following_gpu(inp, r, int(ga[r]), temp)
            assert n_forced >= 1
        assert ga[r] == a_r, f"request {r}: accepted {ga[r]} vs oracle {a_r}"
        draws_checked += 1
        if gn[r] == n_r:
            continue
        assert info_r["draw_gap"] < DRAW_TOL, (
            f"request {r}: drew {gn[r]} vs oracle {n_r} although the oracle's CDF margin is "
            f"{info_r['draw_gap']:.2e} of the total")
        v = int(gn[r])
        w, c, tgt = info_r["weights"], info_r["cdf"], info_r["target"]
        W = c[-1]
        lo = c[v - 1] if v > 0 else 0.0
        assert 0 <= v < len(w), f"request {r}: drew id {v} outside the vocabulary"
        assert w[v] > 0, f"request {r}: drew id {v} of zero weight"
        assert lo - DRAW_TOL * W <= tgt <= c[v] + DRAW_TOL * W, f"request {r}: id {v} outside the CDF step"
    assert ambiguous <= max(1, int(max_ambiguous_frac * R)), f"{ambiguous} ambiguous requests of {R}"
    return draws_checked


@pytest.mark.parametrize("name", ["c0", "c1", "c2", "c3", "c4"])
def test_sampled_configs(sv, name):
    inp = make_sampled_inputs(name, seed=0)
    got = run_gpu(sv, inp)
    assert check_sampled(inp, got) >= 1
    again = run_gpu(sv, inp)  # the workspace counters were left at zero
    for g, h in zip(got, again):
        assert np.array_equal(g, h)


@pytest.mark.parametrize("temperature", [0.5, 2.0])
def test_sampled_temperatures(sv, temperature):
    inp = make_sampled_inputs("c2", seed=3, temperature=temperature)
    check_sampled(inp, run_gpu(sv, inp))


@pytest.mark.parametrize("seed", [11, 12, 13])
def test_sampled_many_requests(sv, seed):
    """Many small requests: a wide spread of accept counts and both draw kinds."""
    cfg = small_config("c2", R=96, k=5, vocab=4096, kv_lens=None, kv_len_range=(100, 200))
    inp = make_sampled_inputs(cfg, seed=seed)
    got = run_gpu(sv, inp)
    check_sampled(inp, got)
    assert len(set(got[0].tolist())) >= 3


@pytest.mark.parametrize("V", [1, 3, 1001, 5000])
def test_sampled_odd_vocab(sv, V):
    """V not a multiple of 4: the scalar load path."""
    cfg = small_config("c0", vocab=V, R=6, k=2, kv_lens=None, kv_len_range=(20, 40))
    inp = make_sampled_inputs(cfg, seed=V)
    check_sampled(inp, run_gpu(sv, inp), max_ambiguous_frac=0.5)


def test_sampled_low_temperature_is_greedy(sv):
    """temperature 1e-3 and one-hot drafts: exactly greedy verification."""
    inp = make_inputs("c2", seed=0)
    R, k = inp["R"], inp["k"]
    V = inp["logits"].shape[1]
    onehot = np.zeros((R, k, V), dtype=np.float32)
    for r in range(R):
        for j in range(k):
            onehot[r, j, inp["draft_tokens"][r][j]] = 1.0
    uni = np.random.default_rng(9).random((R, k + 1)).astype(np.float32) * 0.98 + 0.01
    s_inp = dict(logits=inp["logits"], draft_tokens=inp["draft_tokens"], draft_probs=onehot, uniforms=uni,
                 kv_lens_in=inp["kv_lens_in"], k=k, temperature=1e-3)
    ga, gn, gkv = run_gpu(sv, s_inp)
    _, n, nxt, kv = oracle.ref_greedy_verify(inp["logits"], inp["draft_tokens"], inp["kv_lens_in"], k)
    assert np.array_equal(ga, n) and np.array_equal(gn, nxt) and np.array_equal(gkv, kv)


def test_sampled_draft_equals_target(sv):
    """q = p: every draft is accepted; the bonus token is a draw from p."""
    cfg = small_config("c2", R=8, k=4, vocab=20000, kv_lens=None, kv_len_range=(100, 200))
    inp = make_sampled_inputs(cfg, seed=2)
    k = inp["k"]
    x = inp["logits"].astype(np.float64)
    for r in range(inp["R"]):
        for j in range(k):
            p = np.exp(x[r * (k + 1) + j] - x[r * (k + 1) + j].max())
            inp["draft_probs"][r, j] = (p / p.sum()).astype(np.float32)
    inp["uniforms"][:, :k] = np.minimum(inp["uniforms"][:, :k], 0.999)
    ga, gn, gkv = run_gpu(sv, inp)
    assert np.all(ga == k)
    check_sampled(inp, (ga, gn, gkv))


def test_sampled_zero_residual_falls_back_to_target(sv):
    """q = 2 p everywhere: a rejected draft leaves no residual mass, so the
    next token is drawn from p of the same row."""
    cfg = small_config("c0", R=16, k=3, vocab=3000, kv_lens=None, kv_len_range=(20, 40))
    inp = make_sampled_inputs(cfg, seed=6)
    k = inp["k"]
    x = inp["logits"].astype(np.float64)
    for r in range(inp["R"]):
        for j in range(k):
            p = np.exp(x[r * (k + 1) + j] - x[r * (k + 1) + j].max())
            inp["draft_probs"][r, j] = (2 * p / p.sum()).astype(np.float32)
    # keep the acceptance tests away from u = 0.5
    u = inp["uniforms"]
    u[:, :k] = np.where(np.abs(u[:, :k] - 0.5) < 0.01, 0.3, u[:, :k])
    got = run_gpu(sv, inp)
    assert np.any(got[0] < k)
    check_sampled(inp, got)


def test_sampled_invalid_draft_rejected(sv):
    cfg = small_config("c0", R=4, k=3, vocab=512, kv_lens=None, kv_len_range=(20, 40))
    inp = make_sampled_inputs(cfg, seed=8)
    k = inp["k"]
    inp["draft_probs"][:] = 1.0 / 512
    inp["uniforms"][:, :k] = 0.0  # every in-range draft is accepted (0 < p)
    inp["draft_tokens"][0, 1] = 512
    inp["draft_tokens"][1, 0] = -3
    ga, gn, gkv = run_gpu(sv, inp)
    assert list(ga) == [1, 0, k, k]


@pytest.mark.parametrize("i", range(24))
def test_sampled_sweep(sv, i):
    """Seeded shapes (1-48 requests, k = 0-12, V from 1 to 163840, odd and
    even), temperatures from 0.3 to 3 and draft mixes from nearly one-hot to
    nearly uniform, under the same decision and draw rules."""
    rng = np.random.default_rng(7000 + i)
    R = int(rng.integers(1, 49))
    k = int(rng.integers(0, 13))
    V = int(rng.choice([1, 2, 7, 64, 1000, 4097, 16384, 65536, 163840]))
    while R * (k + 1) * V > 12_000_000:
        R = max(1, R // 2)
    temperature = float(np.exp(rng.uniform(np.log(0.3), np.log(3.0))))
    lo = float(rng.uniform(0.0, 0.9))
    mix = (lo, float(min(1.0, lo + rng.uniform(0.05, 0.5))))
    cfg = small_config("c0", R=R, k=k, vocab=V, kv_lens=None, kv_len_range=(k + 1, 4000))
    inp = make_sampled_inputs(cfg, seed=8000 + i, temperature=temperature, draft_mix=mix)
    got = run_gpu(sv, inp)
    check_sampled(inp, got, max_ambiguous_frac=0.25)
