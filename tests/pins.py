"""Pins for the float64 oracle: checks against things other than the oracle.

Each ``pin_*`` takes the oracle module and raises AssertionError on a
mismatch, so the same pins run against the real oracle (must pass) and
against copies with a planted mistake (must fail; see test_oracle_mutations).

Sources of truth used here, none of them the oracle's own formula:
* a high-accuracy scalar brute force (exactly rounded ``math.fsum`` dot
  products, no max shift, an independent bf16 decode and page walk);
* closed forms (q = 0, identical rows, bound 1, two-row toy, gate limits);
* library routines (scipy.special.logsumexp / softmax / expit);
* invariants (split = unsplit, k = 0 plain decode, page-order invariance,
  (-inf, 0) for bound 0, accepted count range, full-acceptance chain);
* hand-derived greedy cases (argmax ties, acceptance, trim).
"""
from __future__ import annotations

import math
import struct

import numpy as np

from workloads import f32_to_bf16_bits, make_inputs, small_config


# --------------------------------------------------------------------------
# independent helpers
# --------------------------------------------------------------------------
def bf16_to_float(bits: int) -> float:
    return struct.unpack(">f", struct.pack(">I", (int(bits) & 0xFFFF) << 16))[0]


def brute_row(inp, t, h):
    """Scalar brute force for one (token, head): returns (lse, out list)."""
    q_per_req = inp["k"] + 1
    r = t // q_per_req
    ps = inp["page_size"]
    bt = inp["block_table"]
    # walk the pool: which logical position of request r does each page slot hold
    owner = {}
    for i, p in enumerate(bt[r]):
        if p >= 0:
            owner[int(p)] = i
    b = int(inp["kv_bounds"][t])
    rows = [None] * b
    for p, i in owner.items():
        for slot in range(ps):
            j = i * ps + slot
            if j < b:
                rows[j] = [bf16_to_float(x) for x in inp["kv_bits"][p, slot]]
    qv = [bf16_to_float(x) for x in inp["q_bits"][t, h]]
    gv = [bf16_to_float(x) for x in inp["gate_bits"][t, h]]
    D = len(qv)
    if b == 0:
        return -math.inf, [0.0] * D
    scale = inp["softmax_scale"]
    s = [scale * math.fsum(qa * ca for qa, ca in zip(qv, c)) for c in rows]
    e = [math.exp(x) for x in s]
    Z = math.fsum(e)
    o = [math.fsum(e[j] * rows[j][d] for j in range(b)) / Z for d in range(D)]
    out = [o[d] / (1.0 + math.exp(-gv[d])) for d in range(D)]
    return math.log(Z), out


def _toy_inputs(q_rows, kv_rows_list, bounds, gate=None, H=1, k=0, scale=1.0, page_size=4):
    """Explicit tiny inputs (float64 values, D = len(q_rows[0])), one page pool."""
    q = np.asarray(q_rows, dtype=np.float64).reshape(len(bounds), H, -1)
    T, _, D = q.shape
    R = T // (k + 1)
    seqs = [np.asarray(x, dtype=np.float64) for x in kv_rows_list]
    pages = []
    bt_rows = []
    for seq in seqs:
        n_pages = max(1, -(-len(seq) // page_size))
        ids = []
        for i in range(n_pages):
            pg = np.zeros((page_size, D))
            chunk = seq[i * page_size:(i + 1) * page_size]
            pg[:len(chunk)] = chunk
            ids.append(len(pages))
            pages.append(pg)
        bt_rows.append(ids)
    maxp = max(len(x) for x in bt_rows)
    bt = np.full((R, maxp), -1, dtype=np.int32)
    for r, ids in enumerate(bt_rows):
        bt[r, :len(ids)] = ids
    g = np.full((T, H, D), 40.0) if gate is None else np.asarray(gate, dtype=np.float64).reshape(T, H, D)
    return dict(q=q, kv=np.stack(pages), bt=bt, bounds=np.asarray(bounds, dtype=np.int32),
                gate=g, q_per_req=k + 1, scale=scale)


def _run_toy(orc, toy):
    return orc.ref_verify_attention(toy["q"], toy["kv"], toy["bt"], toy["bounds"], toy["gate"],
                                    toy["q_per_req"], toy["scale"])


# --------------------------------------------------------------------------
# attention pins
# --------------------------------------------------------------------------
def pin_bruteforce_c0(orc, heads=(0, 3, 7)):
    inp = make_inputs("c0", seed=0)
    out, lse = orc.ref_verify_attention(inp["q_bits"], inp["kv_bits"], inp["block_table"],
                                        inp["kv_bounds"], inp["gate_bits"], inp["k"] + 1,
                                        inp["softmax_scale"])
    for t in range(inp["T"]):
        for h in heads:
            bl, bo = brute_row(inp, t, h)
            assert abs(lse[t, h] - bl) <= 1e-10 * max(1.0, abs(bl)), (t, h, lse[t, h], bl)
            assert np.allclose(out[t, h], bo, rtol=1e-10, atol=1e-12), (t, h)


def pin_bruteforce_shuffled(orc):
    """Brute force on a small shuffled-pool case with 3 requests and k = 2."""
    cfg = small_config("c0", R=3, k=2, H=2, kv_lens=(5, 130, 64), shuffled=True, vocab=64)
    inp = make_inputs(cfg, seed=3)
    out, lse = orc.ref_verify_attention(inp["q_bits"], inp["kv_bits"], inp["block_table"],
                                        inp["kv_bounds"], inp["gate_bits"], inp["k"] + 1,
                                        inp["softmax_scale"])
    for t in range(inp["T"]):
        for h in range(inp["H"]):
            bl, bo = brute_row(inp, t, h)
            if bl == -math.inf:
                assert lse[t, h] == -math.inf
            else:
                assert abs(lse[t, h] - bl) <= 1e-10 * max(1.0, abs(bl)), (t, h)
            assert np.allclose(out[t, h], bo, rtol=1e-10, atol=1e-12), (t, h)


def pin_two_row_toy(orc):
    """s = (0, ln 3) gives weights (1/4, 3/4): lse = ln 4, o = c0/4 + 3 c1/4."""
    c0 = [0.0, 1.0]
    c1 = [math.log(3.0), 2.0]
    toy = _toy_inputs([[1.0, 0.0]], [[c0, c1]], [2], scale=1.0)
    out, lse = _run_toy(orc, toy)
    sig = 1.0 / (1.0 + math.exp(-40.0))
    assert abs(lse[0, 0] - math.log(4.0)) < 1e-14
    expect = np.array([0.75 * math.log(3.0), 0.25 * 1.0 + 0.75 * 2.0]) * sig
    assert np.allclose(out[0, 0], expect, rtol=1e-14, atol=1e-15)


def pin_closed_forms(orc):
    rng = np.random.default_rng(11)
    D = 8
    seq = rng.standard_normal((9, D))
    # q = 0: every score is 0 -> lse = ln b, o = mean of the visible rows
    toy = _toy_inputs(np.zeros((3, D)), [seq], [1, 5, 9], gate=np.full((3, 1, D), 0.0), k=2)
    out, lse = _run_toy(orc, toy)
    for t, b in enumerate([1, 5, 9]):
        assert abs(lse[t, 0] - math.log(b)) < 1e-13
        assert np.allclose(out[t, 0], 0.5 * seq[:b].mean(axis=0), rtol=1e-13, atol=1e-14)
    # identical visible rows c: o = c, lse = scale <q,c> + ln b
    c = rng.standard_normal(D)
    qv = rng.standard_normal(D)
    toy = _toy_inputs([qv], [np.tile(c, (6, 1))], [6], scale=0.37)
    out, lse = _run_toy(orc, toy)
    sig = 1.0 / (1.0 + math.exp(-40.0))
    assert abs(lse[0, 0] - (0.37 * float(qv @ c) + math.log(6))) < 1e-12
    assert np.allclose(out[0, 0], c * sig, rtol=1e-13)
    # bound 1: o = c_0, lse = s_0
    toy = _toy_inputs([qv], [seq], [1], scale=0.5)
    out, lse = _run_toy(orc, toy)
    assert abs(lse[0, 0] - 0.5 * float(qv @ seq[0])) < 1e-12
    assert np.allclose(out[0, 0], seq[0] * sig, rtol=1e-13)
    # gate 0 halves the output; a large gate passes it through; a very negative one zeroes it
    for gval, factor in ((0.0, 0.5), (60.0, 1.0), (-60.0, 0.0)):
        toy = _toy_inputs([qv], [seq], [4], gate=np.full((1, 1, D), gval), scale=0.5)
        out, _ = _run_toy(orc, toy)
        toy1 = _toy_inputs([qv], [seq], [4], gate=np.full((1, 1, D), 60.0), scale=0.5)
        ref, _ = _run_toy(orc, toy1)
        assert np.allclose(out[0, 0], factor * ref[0, 0], rtol=1e-12, atol=1e-20)


def pin_library_routines(orc):
    """Per-row lse / softmax / sigmoid against scipy's own routines."""
    from scipy.special import expit, logsumexp, softmax
    inp = make_inputs(small_config("c0", R=1, k=1, H=4, kv_lens=(70,)), seed=5)
    out, lse = orc.ref_verify_attention(inp["q_bits"], inp["kv_bits"], inp["block_table"],
                                        inp["kv_bounds"], inp["gate_bits"], 2, inp["softmax_scale"])
    from oracle import bf16_bits_to_f64  # decode only
    q = bf16_bits_to_f64(inp["q_bits"])
    g = bf16_bits_to_f64(inp["gate_bits"])
    kv = bf16_bits_to_f64(inp["kv_bits"]).reshape(-1, inp["D"])  # identity table: page i = positions 64i..
    assert np.array_equal(inp["block_table"][0, :2], [0, 1])
    for t in range(2):
        b = int(inp["kv_bounds"][t])
        C = kv[:b]
        s = inp["softmax_scale"] * (q[t] @ C.T)
        assert np.allclose(lse[t], logsumexp(s, axis=1), rtol=0, atol=1e-12)
        assert np.allclose(out[t], expit(g[t]) * (softmax(s, axis=1) @ C), rtol=1e-12, atol=1e-14)


def pin_zero_bound_identity(orc):
    inp = make_inputs(small_config("c0", R=2, k=1, H=2, kv_lens=(64, 3), vocab=32), seed=2)
    bounds = inp["kv_bounds"].copy()
    bounds[0] = 0
    bounds[3] = 0
    out, lse = orc.ref_verify_attention(inp["q_bits"], inp["kv_bits"], inp["block_table"],
                                        bounds, inp["gate_bits"], 2, inp["softmax_scale"])
    for t in (0, 3):
        assert np.all(lse[t] == -np.inf)
        assert np.all(out[t] == 0.0) and not np.any(np.isnan(out[t]))
    for t in (1, 2):
        assert np.all(np.isfinite(lse[t]))


def pin_split_invariance(orc):
    """Merging split-KV partials equals the unsplit result for any edges."""
    cfg = small_config("c0", R=2, k=3, H=2, kv_lens=(64, 200))
    inp = make_inputs(cfg, seed=4)
    bounds = inp["kv_bounds"].copy()
    bounds[1] = 0
    args = (inp["q_bits"], inp["kv_bits"], inp["block_table"])
    out, lse = orc.ref_verify_attention(*args, bounds, inp["gate_bits"], 4, inp["softmax_scale"])
    for edges in ([[0, 64], [0, 200]], [[0, 30, 64, 64], [0, 64, 128, 200]],
                  [[0, 1, 2, 64], [0, 199, 200, 200]], [[0, 64, 64, 64, 64], [0, 50, 100, 150, 200]]):
        po, pl = orc.ref_attention_partials(*args, bounds, 4, inp["softmax_scale"], edges)
        o2, l2 = orc.ref_lse_combine(po, pl, inp["gate_bits"])
        fin = np.isfinite(lse)
        assert np.array_equal(fin, np.isfinite(l2))
        assert np.allclose(l2[fin], lse[fin], rtol=0, atol=1e-12)
        assert np.allclose(o2, out, rtol=1e-11, atol=1e-13)
        assert not np.any(np.isnan(o2))


def pin_k0_and_single_query(orc):
    """Verify row i with bound b_i equals a plain one-token decode at bound b_i."""
    cfg = small_config("c0", R=2, k=3, H=3, kv_lens=(64, 100))
    inp = make_inputs(cfg, seed=6)
    out, lse = orc.ref_verify_attention(inp["q_bits"], inp["kv_bits"], inp["block_table"],
                                        inp["kv_bounds"], inp["gate_bits"], 4, inp["softmax_scale"])
    for t in range(inp["T"]):
        r = t // 4
        o1, l1 = orc.ref_verify_attention(inp["q_bits"][t:t + 1], inp["kv_bits"],
                                          inp["block_table"][r:r + 1], inp["kv_bounds"][t:t + 1],
                                          inp["gate_bits"][t:t + 1], 1, inp["softmax_scale"])
        assert np.array_equal(l1[0], lse[t]) or np.allclose(l1[0], lse[t], rtol=0, atol=1e-13)
        assert np.allclose(o1[0], out[t], rtol=1e-13, atol=1e-15)


def pin_page_order_invariance(orc):
    """Relabelling pool pages (and the table with them) changes nothing."""
    cfg = small_config("c0", R=2, k=1, H=2, kv_lens=(130, 64))
    inp = make_inputs(cfg, seed=8)
    P = inp["num_pages"]
    perm = np.random.default_rng(1).permutation(P)
    kv2 = np.empty_like(inp["kv_bits"])
    kv2[perm] = inp["kv_bits"]
    bt2 = np.where(inp["block_table"] >= 0, perm[np.maximum(inp["block_table"], 0)], -1)
    a = orc.ref_verify_attention(inp["q_bits"], inp["kv_bits"], inp["block_table"],
                                 inp["kv_bounds"], inp["gate_bits"], 2, inp["softmax_scale"])
    b = orc.ref_verify_attention(inp["q_bits"], kv2, bt2, inp["kv_bounds"], inp["gate_bits"], 2,
                                 inp["softmax_scale"])
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# --------------------------------------------------------------------------
# greedy pins (hand-derived cases; the definitions: argmax with the lowest
# index on ties, accept while d_j == a_{j-1}, kv_out = kv_in - (k - n))
# --------------------------------------------------------------------------
GREEDY_CASES = [
    # name, k, logits rows, drafts, kv_in -> argmax, accepted, next, kv_out
    # rows: [1,3,3,-2] max 3 first at 1; all equal -> 0; [-1,-1,4,4] -> 2.
    # d1 = 1 = a0, d2 = 0 = a1 -> n = 2 = k, next = a2 = 2, kv_out = 10.
    ("ties_full_accept", 2, [[1, 3, 3, -2], [0.5, 0.5, 0.5, 0.5], [-1, -1, 4, 4]], [1, 0], 10,
     [1, 0, 2], 2, 2, 10),
    # a = [3, 0, 1]; d1 = 3 = a0, d2 = 2 != a1 = 0 -> n = 1, next = a1 = 0, kv_out = 20 - 1.
    ("partial_accept", 2, [[0, 0, 0, 9], [5, 4, 3, 2], [0, 7, 7, -7]], [3, 2], 20,
     [3, 0, 1], 1, 0, 19),
    # d1 = 0 != a0 = 2 -> n = 0 although d2 matches a1: only a prefix counts.
    ("first_reject", 2, [[0, 1, 2, -1], [1, 2, 0, 0], [0, 0, 0, 1]], [0, 1], 7,
     [2, 1, 3], 0, 2, 5),
    # k = 0: plain decode, nothing to accept, next = a0, kv unchanged.
    ("k0", 0, [[-3, -1, -2, -1]], [], 5, [1], 0, 1, 5),
    # negative zero and positive zero compare equal: lowest index wins.
    ("signed_zero", 1, [[-0.0, 0.0, -1, -5], [-1, -2, -0.0, 0.0]], [0], 3,
     [0, 2], 1, 2, 3),
]


def pin_greedy_cases(orc):
    for name, k, rows, drafts, kv_in, e_a, e_n, e_next, e_kv in GREEDY_CASES:
        logits = np.asarray(rows, dtype=np.float32)
        d = np.asarray(drafts, dtype=np.int32).reshape(1, k)
        a, n, nxt, kv = orc.ref_greedy_verify(logits, d, np.array([kv_in], dtype=np.int32), k)
        assert list(a) == e_a, (name, list(a))
        assert int(n[0]) == e_n, (name, n)
        assert int(nxt[0]) == e_next, (name, nxt)
        assert int(kv[0]) == e_kv, (name, kv)


def pin_greedy_invariants(orc):
    for cfg_name in ("c0",):
        inp = make_inputs(cfg_name, seed=0)
        k = inp["k"]
        a, n, nxt, kv = orc.ref_greedy_verify(inp["logits"], inp["draft_tokens"], inp["kv_lens_in"], k)
        # the generator planted each row's maximum
        assert np.array_equal(a, inp["planted_argmax"])
        assert np.all((n >= 0) & (n <= k))
        assert np.array_equal(kv, inp["kv_lens_in"] - (k - n))
        # drafts equal to the target argmax chain: everything is accepted
        R = inp["R"]
        chain = np.stack([a[r * (k + 1):r * (k + 1) + k] for r in range(R)])
        a2, n2, nxt2, kv2 = orc.ref_greedy_verify(inp["logits"], chain, inp["kv_lens_in"], k)
        assert np.all(n2 == k) and np.array_equal(kv2, inp["kv_lens_in"])
        assert np.array_equal(nxt2, a[np.arange(R) * (k + 1) + k])
        # first draft wrong: nothing accepted
        bad = chain.copy()
        bad[:, 0] = (chain[:, 0] + 1) % inp["cfg"].vocab
        _, n3, nxt3, kv3 = orc.ref_greedy_verify(inp["logits"], bad, inp["kv_lens_in"], k)
        assert np.all(n3 == 0) and np.array_equal(nxt3, a[np.arange(R) * (k + 1)])
        assert np.array_equal(kv3, inp["kv_lens_in"] - k)


ALL_PINS = [
    pin_bruteforce_c0, pin_bruteforce_shuffled, pin_two_row_toy, pin_closed_forms,
    pin_library_routines, pin_zero_bound_identity, pin_split_invariance,
    pin_k0_and_single_query, pin_page_order_invariance, pin_greedy_cases, pin_greedy_invariants,
]


def bf16_round_cases():
    """(float32 value, expected bf16 bits) for the generator's rounding."""
    return [
        (1.0, 0x3F80),
        (1.0 + 2.0 ** -8, 0x3F80),          # exact tie -> even (down)
        (1.0 + 3 * 2.0 ** -8, 0x3F82),      # tie -> even (up)
        (1.0 + 2.0 ** -8 + 2.0 ** -20, 0x3F81),
        (-2.5, 0xC020),
        (0.0, 0x0000),
    ]


def check_bf16_rounding():
    for v, bits in bf16_round_cases():
        got = int(f32_to_bf16_bits(np.array([v], dtype=np.float32))[0])
        assert got == bits, (v, hex(got), hex(bits))


# --------------------------------------------------------------------------
# KV append pins: the definition is a scatter, so the pins are properties that
# do not restate it: read-back through the independent page walk, untouched
# rows, skipped tokens, and page-order invariance.
# --------------------------------------------------------------------------
def pin_kv_append(orc):
    cfg = small_config("c0", R=3, k=2, H=2, kv_lens=(5, 130, 64), shuffled=True, vocab=64)
    inp = make_inputs(cfg, seed=9)
    k1 = inp["k"] + 1
    rng = np.random.default_rng(9)
    T = inp["T"]
    kv_new = f32_to_bf16_bits(rng.standard_normal((T, inp["D"]), dtype=np.float32))
    # verify-group positions L-k-1 .. L-1; the middle token of request 1 is skipped
    pos = np.concatenate([np.arange(L - k1, L) for L in inp["kv_lens_in"]]).astype(np.int32)
    pos[k1 + 1] = -1
    pool = orc.ref_kv_append(inp["kv_bits"], inp["block_table"], pos, kv_new, k1)
    # read back through an inverse page walk (independent of the scatter)
    owner = {}
    for r in range(inp["R"]):
        for i, p in enumerate(inp["block_table"][r]):
            if p >= 0:
                owner[int(p)] = (r, i)
    written = set()
    for t in range(T):
        if pos[t] < 0:
            continue
        r = t // k1
        hits = [(p, s) for p, (rr, i) in owner.items() if rr == r for s in range(64) if i * 64 + s == pos[t]]
        assert len(hits) == 1
        p, s = hits[0]
        assert np.array_equal(pool[p, s], kv_new[t])
        written.add((p, s))
    # everything else is untouched, including the skipped token's slot
    for p in range(pool.shape[0]):
        for s in range(64):
            if (p, s) not in written:
                assert np.array_equal(pool[p, s], inp["kv_bits"][p, s])
    assert len(written) == T - 1
    # relabelling the pages commutes with the append
    perm = np.random.default_rng(2).permutation(pool.shape[0])
    kv2 = np.empty_like(inp["kv_bits"]); kv2[perm] = inp["kv_bits"]
    bt2 = np.where(inp["block_table"] >= 0, perm[np.maximum(inp["block_table"], 0)], -1)
    pool2 = orc.ref_kv_append(kv2, bt2, pos, kv_new, k1)
    assert np.array_equal(pool2[perm], pool)


ALL_PINS.append(pin_kv_append)


# --------------------------------------------------------------------------
# sampled (rejection-sampling) verification
# --------------------------------------------------------------------------
# Pins independent of the oracle's formulas: the defining property of
# speculative sampling (every emitted token is distributed as the target
# distribution, whatever the draft distribution), checked by Monte Carlo with a
# chi-square test; hand-derived accept/reject and draw cases; scipy's softmax;
# the closed form q = p (every draft accepted); and the low-temperature limit,
# where sampled verification with one-hot drafts must equal greedy
# verification.
def _mc_emitted(orc, p_rows, q_rows, trials, seed):
    """Run the oracle on `trials` independent draws of (drafts ~ q, uniforms)
    and return the emitted tokens per position (-1 where not emitted)."""
    rng = np.random.default_rng(seed)
    k = q_rows.shape[0]
    V = p_rows.shape[1]
    logits = np.log(p_rows).astype(np.float64)
    R = trials
    drafts = np.stack([rng.choice(V, size=R, p=q_rows[j]) for j in range(k)], axis=1)
    uni = rng.random((R, k + 1))
    a, nxt, _ = orc.ref_sampled_verify(np.tile(logits, (R, 1)), drafts, np.tile(q_rows, (R, 1, 1)),
                                       uni, np.full(R, 100), k, 1.0)
    emitted = np.full((R, k + 1), -1, dtype=np.int64)
    for r in range(R):
        n = int(a[r])
        emitted[r, :n] = drafts[r, :n]
        emitted[r, n] = nxt[r]
    return emitted


def _chi2_ok(samples, p, alpha=1e-6):
    from scipy.stats import chisquare
    counts = np.bincount(samples, minlength=len(p)).astype(np.float64)
    expected = p * counts.sum()
    keep = expected > 0
    assert counts[~keep].sum() == 0, "a token of zero target probability was emitted"
    return chisquare(counts[keep], expected[keep]).pvalue > alpha


def pin_sampled_distribution(orc):
    """Each emitted position is distributed as the target row it verifies."""
    p = np.array([[0.40, 0.25, 0.15, 0.10, 0.06, 0.04],
                  [0.05, 0.05, 0.50, 0.10, 0.20, 0.10],
                  [0.30, 0.30, 0.10, 0.10, 0.10, 0.10]])
    q = np.array([[0.05, 0.50, 0.05, 0.30, 0.05, 0.05],
                  [0.30, 0.10, 0.10, 0.10, 0.30, 0.10]])
    em = _mc_emitted(orc, p, q, trials=6000, seed=123)
    assert _chi2_ok(em[:, 0], p[0]), "first emitted token is not distributed as p_0"
    sel = em[:, 1] >= 0
    assert sel.sum() > 1000 and _chi2_ok(em[sel, 1], p[1]), "second emitted token is not p_1"
    sel = em[:, 2] >= 0
    assert sel.sum() > 300 and _chi2_ok(em[sel, 2], p[2]), "bonus token is not p_2"


def pin_sampled_hand_cases(orc):
    p = np.array([0.5, 0.3, 0.2])
    q = np.array([[0.2, 0.7, 0.1]])
    x = np.log(p)[None, :].repeat(2, axis=0)

    def run(u0, u1):
        a, nxt, kv = orc.ref_sampled_verify(x, [[1]], q[None], np.array([[u0, u1]]), [50], 1, 1.0)
        return int(a[0]), int(nxt[0]), int(kv[0])
    # accept iff u * 0.7 < 0.3, i.e. u < 3/7 = 0.42857...
    assert run(0.42, 0.5)[0] == 1
    assert run(0.43, 0.5)[0] == 0
    # rejected: residual max(0, p - q) = [0.3, 0, 0.1], total 0.4
    assert run(0.43, 0.74) == (0, 0, 49)   # 0.74 * 0.4 = 0.296 < 0.3
    assert run(0.43, 0.76) == (0, 2, 49)   # 0.304 > 0.3: skips the zero-weight id 1
    # accepted: the bonus token is drawn from p of the last verify token
    assert run(0.1, 0.49) == (1, 0, 50)
    assert run(0.1, 0.51) == (1, 1, 50)
    assert run(0.1, 0.81) == (1, 2, 50)
    # inverse CDF on its own
    assert orc.inverse_cdf(np.array([1.0, 0.0, 3.0]), 0.2) == 0
    assert orc.inverse_cdf(np.array([1.0, 0.0, 3.0]), 0.25) == 2
    assert orc.inverse_cdf(np.array([0.0, 0.0, 5.0]), 0.0) == 2
    assert orc.inverse_cdf(np.array([2.0, 2.0]), 0.0) == 0


def pin_sampled_closed_forms(orc):
    from scipy.special import softmax
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 40)) * 2
    for temp in (0.5, 1.0, 3.0):
        assert np.allclose(orc.target_probs(x[0], temp), softmax(x[0] / temp), rtol=1e-12, atol=0)
    # q = p at every position: every draft is accepted, whatever u < 1
    k, R = 2, 50
    temp = 0.7
    xs = rng.standard_normal((R * (k + 1), 40))
    qp = np.stack([np.stack([softmax(xs[r * (k + 1) + j] / temp) for j in range(k)]) for r in range(R)])
    drafts = rng.integers(0, 40, size=(R, k))
    uni = rng.random((R, k + 1)) * 0.999999
    a, nxt, kv = orc.ref_sampled_verify(xs, drafts, qp, uni, np.full(R, 10), k, temp)
    assert np.all(a == k) and np.all(kv == 10)


def pin_sampled_greedy_limit(orc):
    """Low temperature + one-hot drafts = greedy verification."""
    inp = make_inputs(small_config("c0", vocab=512), seed=4)
    R, k = inp["R"], inp["k"]
    V = inp["logits"].shape[1]
    a_g, n_g, nxt_g, kv_g = orc.ref_greedy_verify(inp["logits"], inp["draft_tokens"], inp["kv_lens_in"], k)
    onehot = np.zeros((R, k, V))
    for r in range(R):
        for j in range(k):
            onehot[r, j, inp["draft_tokens"][r][j]] = 1.0
    uni = np.random.default_rng(1).random((R, k + 1)) * 0.98 + 0.01
    a, nxt, kv = orc.ref_sampled_verify(inp["logits"], inp["draft_tokens"], onehot, uni, inp["kv_lens_in"],
                                        k, 1e-3)
    assert np.array_equal(a, n_g) and np.array_equal(nxt, nxt_g) and np.array_equal(kv, kv_g)


SAMPLED_PINS = [pin_sampled_distribution, pin_sampled_hand_cases, pin_sampled_closed_forms,
                pin_sampled_greedy_limit]


# --------------------------------------------------------------------------
# head-wise gate and the W_UV value up-projection
# --------------------------------------------------------------------------
def pin_headwise_gate(orc):
    """A [T, H] gate scales whole latent rows: brute force on sampled rows,
    the gate-0 closed form (half the ungated output) and equality with the
    same values broadcast over the 512 columns."""
    inp = make_inputs("c0", seed=0)
    k1 = inp["k"] + 1
    g_head = inp["gate_bits"][:, :, 0].copy()  # bf16 bits [T, H]
    out_hw, lse_hw = orc.ref_verify_attention(inp["q_bits"], inp["kv_bits"], inp["block_table"],
                                              inp["kv_bounds"], g_head, k1, inp["softmax_scale"])
    for t, h in ((0, 0), (5, 3), (7, 7)):
        b = dict(inp)
        b["gate_bits"] = np.repeat(g_head[:, :, None], inp["gate_bits"].shape[2], axis=2)
        lse_b, out_b = brute_row(b, t, h)
        assert abs(lse_hw[t, h] - lse_b) < 1e-9
        assert np.allclose(out_hw[t, h], out_b, rtol=1e-9, atol=1e-12)
    zero = np.zeros_like(g_head)
    out0, _ = orc.ref_verify_attention(inp["q_bits"], inp["kv_bits"], inp["block_table"], inp["kv_bounds"],
                                       zero, k1, inp["softmax_scale"])
    big = np.full(inp["gate_bits"].shape, 60.0)
    out_ungated, _ = orc.ref_verify_attention(inp["q_bits"], inp["kv_bits"], inp["block_table"],
                                              inp["kv_bounds"], big, k1, inp["softmax_scale"])
    assert np.allclose(out0, 0.5 * out_ungated, rtol=1e-12, atol=1e-14)
    # the merge applies the head-wise gate the same way
    po, pl = orc.ref_attention_partials(inp["q_bits"], inp["kv_bits"], inp["block_table"], inp["kv_bounds"], k1,
                                        inp["softmax_scale"], [[0, 40, 100], [0, 30, 100]])
    om, lm = orc.ref_lse_combine(po, pl, g_head)
    assert np.allclose(om, out_hw, rtol=1e-9, atol=1e-12)
    fin = np.isfinite(lse_hw)
    assert np.array_equal(np.isfinite(lm), fin) and np.allclose(lm[fin], lse_hw[fin], rtol=0, atol=1e-9)


def pin_wuv_projection(orc):
    """v[t, h] = W_UV[h] @ out[t, h]: scalar brute force (exactly rounded
    sums), the identity projection, and commuting with a head-wise gate."""
    rng = np.random.default_rng(31)
    T, H, D, V = 3, 4, 512, 16
    x = rng.standard_normal((T, H, D))
    w = rng.standard_normal((H, V, D))
    v = orc.ref_wuv_project(x, w)
    assert v.shape == (T, H, V)
    for t in range(T):
        for h in range(H):
            for j in (0, 7, V - 1):
                ref = math.fsum(float(w[h, j, d]) * float(x[t, h, d]) for d in range(D))
                assert abs(v[t, h, j] - ref) < 1e-10
    eye = np.broadcast_to(np.eye(D), (H, D, D))
    assert np.allclose(orc.ref_wuv_project(x, eye), x, rtol=0, atol=1e-12)
    # bf16 bit inputs widen exactly
    xb = f32_to_bf16_bits(x.astype(np.float32))
    wb = f32_to_bf16_bits(w.astype(np.float32))
    vb = orc.ref_wuv_project(xb, wb)
    xf = np.array([[[bf16_to_float(a) for a in row] for row in m] for m in xb[:1, :1]])
    wf = np.array([[bf16_to_float(a) for a in row] for row in wb[0, :2]])
    assert abs(vb[0, 0, 1] - math.fsum(float(p) * float(q) for p, q in zip(wf[1], xf[0, 0]))) < 1e-9
    # a head-wise gate commutes with the projection
    g = rng.standard_normal((T, H))
    sg = 1.0 / (1.0 + np.exp(-g))
    assert np.allclose(orc.ref_wuv_project(sg[..., None] * x, w), sg[..., None] * v, rtol=1e-12, atol=1e-12)


ALL_PINS += [pin_headwise_gate, pin_wuv_projection]


# --------------------------------------------------------------------------
# fp8 latent KV
# --------------------------------------------------------------------------
def pin_e4m3_decode(orc):
    """The E4M3 decode against torch's float8_e4m3fn for all 256 codes, plus
    hand values (largest normal 448, smallest subnormal 2^-9, NaN codes)."""
    import torch
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    got = orc.e4m3_bits_to_f64(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert orc.e4m3_bits_to_f64(np.array([0x7E]))[0] == 448.0
    assert orc.e4m3_bits_to_f64(np.array([0x01]))[0] == 2.0 ** -9
    assert orc.e4m3_bits_to_f64(np.array([0xB8]))[0] == -1.0
    assert orc.e4m3_bits_to_f64(np.array([0x80]))[0] == 0.0


def pin_fp8_attention_scale(orc):
    """Attention over an fp8 pool is the attention over its dequantised rows;
    the pool scale only rescales the scores and the output: with kv_scale s,
    (softmax_scale, s) gives the same lse as (softmax_scale * s, 1) and s times
    its output."""
    inp = make_inputs("c0", seed=1)
    from workloads import fp8_kv_pool
    codes, s = fp8_kv_pool(inp)
    k1 = inp["k"] + 1
    deq = orc.e4m3_bits_to_f64(codes) * s
    o1, l1 = orc.ref_verify_attention(inp["q_bits"], deq, inp["block_table"], inp["kv_bounds"],
                                      inp["gate_bits"], k1, inp["softmax_scale"])
    o2, l2 = orc.ref_verify_attention(inp["q_bits"], orc.e4m3_bits_to_f64(codes), inp["block_table"],
                                      inp["kv_bounds"], inp["gate_bits"], k1, inp["softmax_scale"] * s)
    fin = np.isfinite(l1)
    assert np.array_equal(fin, np.isfinite(l2))
    assert np.allclose(l1[fin], l2[fin], rtol=0, atol=1e-9)
    assert np.allclose(o1, s * o2, rtol=1e-9, atol=1e-12)
    # the quantised pool stays close to the bf16 one (|error| <= 2^-4 relative + subnormal step)
    bf = orc.bf16_bits_to_f64(inp["kv_bits"])
    assert np.all(np.abs(deq - bf) <= np.abs(bf) / 16 + s * 2.0 ** -10)


ALL_PINS += [pin_e4m3_decode, pin_fp8_attention_scale]
