"""GPU parity: the CUDA path, called through the C ABI, against the float64
oracle on the same seeded inputs.  Integer outputs must match bit for bit;
floating outputs within the tolerances in gpu_util."""
import numpy as np
import pytest
import torch

import oracle
import pins
from gpu_util import bf16_tensor, check_attention, device_inputs, i32, to_f64
from workloads import CONFIGS, make_inputs, small_config

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verify_mla_gb300 as m
    m.load_library()
    return m


_cache = {}


def inputs_for(name, seed=0):
    key = (name, seed)
    if key not in _cache:
        _cache[key] = make_inputs(name, seed=seed)
    return _cache[key]


def run_attention(sv, inp, num_splits=0, kv_bits=None, bounds=None, status=None):
    d = device_inputs(inp, DEV)
    kv = d["kv"] if kv_bits is None else bf16_tensor(kv_bits, DEV)
    kb = d["kv_bounds"] if bounds is None else i32(bounds, DEV)
    out, lse = sv.mla_verify_decode(d["q"], kv, d["block_table"], kb, d["gate"], inp["k"] + 1,
                                    inp["softmax_scale"], num_splits=num_splits, status=status)
    torch.cuda.synchronize()
    return out, lse


def oracle_attention(inp, bounds=None, kv_bits=None):
    return oracle.ref_verify_attention(inp["q_bits"], inp["kv_bits"] if kv_bits is None else kv_bits,
                                       inp["block_table"],
                                       inp["kv_bounds"] if bounds is None else bounds,
                                       inp["gate_bits"], inp["k"] + 1, inp["softmax_scale"])


# ----------------------------------------------------------------- greedy
@pytest.mark.parametrize("name", ["c0", "c1", "c2", "c3", "c4"])
def test_greedy_configs_bit_exact(sv, name):
    inp = inputs_for(name)
    d = device_inputs(inp, DEV)
    a, n, nxt, kv = oracle.ref_greedy_verify(inp["logits"], inp["draft_tokens"], inp["kv_lens_in"], inp["k"])
    for _ in range(2):  # the second call checks the workspace was left zeroed
        ga, gn, gnxt, gkv = sv.spec_verify_greedy(d["logits"], d["draft_tokens"], d["kv_lens_in"], inp["k"])
        torch.cuda.synchronize()
        assert np.array_equal(ga.cpu().numpy(), a)
        assert np.array_equal(gn.cpu().numpy(), n)
        assert np.array_equal(gnxt.cpu().numpy(), nxt)
        assert np.array_equal(gkv.cpu().numpy(), kv)


@pytest.mark.parametrize("R,k,V,p", [(3, 40, 3000, 0.97), (1, 63, 163840, 0.99), (200, 1, 5000, 0.5)])
def test_greedy_group_sizes(sv, R, k, V, p):
    """Long verify groups (k + 1 > 32, drafts matching with high probability
    so that long prefixes are accepted) and many short ones, against the oracle."""
    cfg = small_config("c0", R=R, k=k, H=1, vocab=V, draft_p=p, kv_lens=None, kv_len_range=(k + 2, k + 300))
    inp = make_inputs(cfg, seed=R + k)
    d = device_inputs(inp, DEV)
    a, n, nxt, kv = oracle.ref_greedy_verify(inp["logits"], inp["draft_tokens"], inp["kv_lens_in"], k)
    ga, gn, gnxt, gkv = sv.spec_verify_greedy(d["logits"], d["draft_tokens"], d["kv_lens_in"], k)
    torch.cuda.synchronize()
    assert np.array_equal(ga.cpu().numpy(), a)
    assert np.array_equal(gn.cpu().numpy(), n)
    assert np.array_equal(gnxt.cpu().numpy(), nxt)
    assert np.array_equal(gkv.cpu().numpy(), kv)
    assert n.min() >= 0 and n.max() <= k


def _greedy_case(sv, logits, drafts, kv_in, k):
    lt = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).to(DEV)
    dt = torch.from_numpy(np.ascontiguousarray(np.asarray(drafts, dtype=np.int32).reshape(len(kv_in), k))).to(DEV)
    kt = torch.from_numpy(np.asarray(kv_in, dtype=np.int32)).to(DEV)
    res = sv.spec_verify_greedy(lt, dt, kt, k)
    torch.cuda.synchronize()
    return [r.cpu().numpy() for r in res]


def test_greedy_hand_cases(sv):
    for name, k, rows, drafts, kv_in, e_a, e_n, e_next, e_kv in pins.GREEDY_CASES:
        a, n, nxt, kv = _greedy_case(sv, np.asarray(rows, dtype=np.float32), drafts, [kv_in], k)
        assert list(a) == e_a, name
        assert int(n[0]) == e_n and int(nxt[0]) == e_next and int(kv[0]) == e_kv, name


@pytest.mark.parametrize("V", [1, 3, 4, 1000, 4099, 163840, 200003])
def test_greedy_ties_across_chunks(sv, V):
    rng = np.random.default_rng(V)
    R, k = 3, 2
    T = R * (k + 1)
    x = rng.standard_normal((T, V)).astype(np.float32)
    for t in range(T):
        pos = np.sort(rng.choice(V, size=min(V, 3), replace=False))
        x[t, pos] = 50.0  # the same maximum at several places, far apart
    x[0, :] = -0.0
    if V > 1:
        x[0, V - 1] = 0.0  # +0 after -0: still the lowest index wins
    drafts = rng.integers(0, V, size=(R, k)).astype(np.int32)
    kv_in = rng.integers(10, 100, size=R).astype(np.int32)
    ref = oracle.ref_greedy_verify(x, drafts, kv_in, k)
    got = _greedy_case(sv, x, drafts, kv_in, k)
    for g, r in zip(got, ref):
        assert np.array_equal(g, r)


def test_greedy_full_chain_and_first_reject(sv):
    inp = inputs_for("c1")
    k = inp["k"]
    a = inp["planted_argmax"]
    chain = a[:k].reshape(1, k)
    got = _greedy_case(sv, inp["logits"], chain, inp["kv_lens_in"], k)
    assert int(got[1][0]) == k and int(got[3][0]) == int(inp["kv_lens_in"][0])
    bad = chain.copy()
    bad[0, 0] = (bad[0, 0] + 1) % inp["cfg"].vocab
    got = _greedy_case(sv, inp["logits"], bad, inp["kv_lens_in"], k)
    assert int(got[1][0]) == 0 and int(got[2][0]) == int(a[0])
    assert int(got[3][0]) == int(inp["kv_lens_in"][0]) - k


# ----------------------------------------------------------------- combine
@pytest.mark.parametrize("edges_kind", ["even", "with_empty"])
def test_combine_matches_oracle(sv, edges_kind):
    cfg = small_config("c0", R=2, k=3, H=16, kv_lens=(150, 260))
    inp = make_inputs(cfg, seed=1)
    bounds = inp["kv_bounds"].copy()
    bounds[2] = 0
    if edges_kind == "even":
        edges = [[0, 50, 100, 150], [0, 90, 180, 260]]
    else:
        edges = [[0, 150, 150, 150], [0, 0, 200, 260]]
    po, pl = oracle.ref_attention_partials(inp["q_bits"], inp["kv_bits"], inp["block_table"], bounds, 4,
                                           inp["softmax_scale"], edges)
    ref_o, ref_l = oracle.ref_lse_combine(po, pl, inp["gate_bits"])
    pot = torch.from_numpy(po.astype(np.float32)).to(DEV)
    plt = torch.from_numpy(pl.astype(np.float32)).to(DEV)
    out, lse = sv.mla_lse_combine(pot, plt, bf16_tensor(inp["gate_bits"], DEV))
    torch.cuda.synchronize()
    check_attention(out, lse, ref_o, ref_l, label="combine")


# ----------------------------------------------------------------- attention
@pytest.mark.parametrize("name", ["c0", "c1", "c2", "c3"])
def test_attention_configs(sv, name):
    inp = inputs_for(name)
    ref_o, ref_l = oracle_attention(inp)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = run_attention(sv, inp, status=status)
    assert int(status.item()) == 0
    check_attention(out, lse, ref_o, ref_l, label=name)


def test_attention_c4_full(sv):
    """The full-size long-context workload (16 requests, contexts 8K-32K,
    straddling groups, 10% zero bounds; the balanced split plan cuts every
    request into pieces) against the oracle on every token and head."""
    inp = inputs_for("c4")
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = run_attention(sv, inp, status=status)
    assert int(status.item()) == 0
    ref_o, ref_l = oracle_attention(inp)
    check_attention(out, lse, ref_o, ref_l, label="c4 full")
    # the zero-bound tokens give exactly (-inf, 0), every other row is finite
    l = to_f64(lse)
    pos = inp["kv_bounds"] > 0
    assert (~pos).sum() == len(inp["zero_bound_tokens"]) > 0
    assert np.all(np.isfinite(l[pos])) and np.all(l[~pos] == -np.inf)


def _mid_config(**kw):
    base = dict(R=3, k=4, H=64, kv_lens=(70, 700, 333), shuffled=True, vocab=64)
    base.update(kw)
    return small_config("c2", kv_len_range=None, **base)


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64])
def test_attention_split_sweep(sv, splits):
    inp = make_inputs(_mid_config(), seed=2)
    ref_o, ref_l = oracle_attention(inp)
    out, lse = run_attention(sv, inp, num_splits=splits)
    check_attention(out, lse, ref_o, ref_l, label=f"splits={splits}")


def test_attention_longest_context(sv):
    """One request of 131072 positions (2048 KV tiles, k = 3, H = 16: 64
    rows): the automatic uniform split, and the balanced plan in both forms,
    where the piece length reaches its lower bound ceil(n_r / SV_MAX_SPLITS)
    (64 pieces of 32 tiles); every token and head against the oracle."""
    cfg = small_config("c0", R=1, k=3, H=16, kv_lens=(131072,), kv_len_range=None, shuffled=True, vocab=64)
    inp = make_inputs(cfg, seed=7)
    ref_o, ref_l = oracle_attention(inp)
    d = device_inputs(inp, DEV)
    for splits, form in ((0, sv.FORM_AUTO), (sv.SV_SPLITS_BALANCED, sv.FORM_STACKED),
                         (sv.SV_SPLITS_BALANCED, sv.FORM_TWO_CTA)):
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        out, lse = sv.mla_verify_decode(d["q"], d["kv"], d["block_table"], d["kv_bounds"], d["gate"], 4,
                                        inp["softmax_scale"], num_splits=splits, status=status, form=form)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        check_attention(out, lse, ref_o, ref_l, label=f"131072 positions, splits={splits}, form={form}")


@pytest.mark.parametrize("q_factor", [0.0, 16.0, 64.0])
def test_attention_extreme_scores(sv, q_factor):
    """A zero query (every visible row weighs the same: o is the mean of the
    rows, lse = ln b) and a query scaled by 16 or 64 (scores spread over
    hundreds of log2 units, so the running maximum moves again and again and
    nearly all of each row's weight sits on a few KV rows), in every split
    mode: the lazy rescale and the merge against the float64 oracle."""
    cfg = small_config("c0", R=3, k=3, H=16, kv_lens=(2000, 700, 129), kv_len_range=None, shuffled=True,
                       vocab=64)
    inp = make_inputs(cfg, seed=17)
    from workloads import f32_to_bf16_bits
    q = inp["q_bits"].astype(np.uint32) << 16
    q = f32_to_bf16_bits(q.view(np.float32) * np.float32(q_factor))
    inp = dict(inp, q_bits=q)
    ref_o, ref_l = oracle_attention(inp)
    d = device_inputs(inp, DEV)
    for splits in (1, 3, sv.SV_SPLITS_BALANCED):
        for form in (sv.FORM_TWO_CTA, sv.FORM_STACKED):
            status = torch.zeros(1, dtype=torch.int32, device=DEV)
            out, lse = sv.mla_verify_decode(d["q"], d["kv"], d["block_table"], d["kv_bounds"], d["gate"], 4,
                                            inp["softmax_scale"], num_splits=splits, status=status, form=form)
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            check_attention(out, lse, ref_o, ref_l, label=f"q x {q_factor}, splits={splits}, form={form}")


def test_attention_wave_mode(sv):
    """The wave split mode (the first k requests whole, the others in s
    pieces) on 30 requests x 3 row tiles x 2 halves = 180 CTAs: ragged
    contexts, zero bounds in whole and in split requests, NaN pool slack,
    both gate shapes."""
    rng = np.random.default_rng(21)
    lens = tuple(int(x) for x in rng.integers(70, 700, size=30))
    cfg = small_config("c2", R=30, k=4, H=64, kv_lens=lens, kv_len_range=None, shuffled=True, vocab=64)
    inp = make_inputs(cfg, seed=21)
    assert sv.num_splits_for(inp["R"], 5, 64, inp["max_pages"]) == sv.SV_SPLITS_WAVE
    bounds = inp["kv_bounds"].copy()
    bounds[[0, 3, 5 * 28 + 1, 5 * 29 + 4]] = 0  # whole requests 0 and 28's neighbours, split requests too
    kv = inp["kv_bits"].copy()
    for r in range(inp["R"]):
        L = int(inp["kv_lens_in"][r])
        kv[int(inp["block_table"][r, (L - 1) // 64]), L % 64 if L % 64 else 64:] = 0x7FC0
    ref_o, ref_l = oracle_attention(inp, bounds=bounds, kv_bits=kv)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = run_attention(sv, inp, num_splits=sv.SV_SPLITS_WAVE, kv_bits=kv, bounds=bounds, status=status)
    assert int(status.item()) == 0
    check_attention(out, lse, ref_o, ref_l, label="wave mode")
    g_head = np.ascontiguousarray(inp["gate_bits"][:, :, 0])
    ref_oh, ref_lh = oracle.ref_verify_attention(inp["q_bits"], kv, inp["block_table"], bounds, g_head, 5,
                                                 inp["softmax_scale"])
    d = device_inputs(inp, DEV)
    out_h, lse_h = sv.mla_verify_decode(d["q"], bf16_tensor(kv, DEV), d["block_table"], i32(bounds, DEV),
                                        bf16_tensor(g_head, DEV), 5, inp["softmax_scale"],
                                        num_splits=sv.SV_SPLITS_WAVE)
    torch.cuda.synchronize()
    check_attention(out_h, lse_h, ref_oh, ref_lh, label="wave mode, head-wise gate")


def test_attention_partials_layout(sv):
    """The split partials in the workspace follow the documented layout and
    equal the oracle's partials over the documented tile ranges."""
    inp = make_inputs(_mid_config(), seed=3)
    S = 3
    d = device_inputs(inp, DEV)
    T, H = inp["T"], inp["H"]
    ws = torch.empty(sv.attention_workspace_bytes(T, H, S), dtype=torch.uint8, device=DEV)
    sv.mla_verify_decode(d["q"], d["kv"], d["block_table"], d["kv_bounds"], d["gate"], inp["k"] + 1,
                         inp["softmax_scale"], num_splits=S, workspace=ws)
    torch.cuda.synchronize()
    n_o = S * T * H * 512
    part_o = ws[:2 * n_o].view(torch.bfloat16).view(S, T, H, 512)
    part_lse = ws[2 * n_o:2 * n_o + 4 * S * T * H].view(torch.float32).view(S, T, H)
    k1 = inp["k"] + 1
    edges = []
    for r in range(inp["R"]):
        n_r = -(-int(inp["kv_bounds"][r * k1:(r + 1) * k1].max()) // 64)
        edges.append([min(64 * ((s * n_r) // S), 10 ** 9) for s in range(S + 1)])
    po, pl = oracle.ref_attention_partials(inp["q_bits"], inp["kv_bits"], inp["block_table"], inp["kv_bounds"],
                                           k1, inp["softmax_scale"], edges)
    gl = to_f64(part_lse)
    assert np.array_equal(np.isfinite(gl), np.isfinite(pl))
    fin = np.isfinite(pl)
    assert np.max(np.abs(gl[fin] - pl[fin])) <= 1e-3
    go = to_f64(part_o)
    assert np.linalg.norm(go - po) / np.linalg.norm(po) <= 1e-2
    assert np.all(go[~fin] == 0.0)


def test_zero_bound_rows(sv):
    inp = make_inputs(_mid_config(), seed=4)
    bounds = inp["kv_bounds"].copy()
    k1 = inp["k"] + 1
    bounds[0] = 0
    bounds[k1:2 * k1] = 0  # a whole request fully masked
    bounds[2 * k1 + 3] = 0
    ref_o, ref_l = oracle_attention(inp, bounds=bounds)
    for splits in (1, 4):
        out, lse = run_attention(sv, inp, num_splits=splits, bounds=bounds)
        check_attention(out, lse, ref_o, ref_l, label=f"zero bounds, splits={splits}")


def test_nan_in_pool_slack_does_not_leak(sv):
    inp = make_inputs(_mid_config(), seed=5)
    kv = inp["kv_bits"].copy()
    bt = inp["block_table"]
    for r in range(inp["R"]):
        L = int(inp["kv_lens_in"][r])
        last = int(bt[r, (L - 1) // 64])
        kv[last, L % 64 if L % 64 else 64:] = 0x7FC0  # NaN beyond the request's last row
    ref_o, ref_l = oracle_attention(inp, kv_bits=kv)
    for splits in (1, 3):
        out, lse = run_attention(sv, inp, num_splits=splits, kv_bits=kv)
        check_attention(out, lse, ref_o, ref_l, label=f"nan slack, splits={splits}")


@pytest.mark.parametrize("H,k,lens", [(96, 1, (300, 129)), (1, 0, (65, 1, 640)), (8, 19, (500,)), (64, 7, (64,)),
                                      (3, 40, (700, 300)), (8, 35, (900,)), (128, 15, (1500, 700))])
def test_attention_head_and_group_shapes(sv, H, k, lens):
    cfg = small_config("c0", R=len(lens), k=k, H=H, kv_lens=lens, shuffled=True, vocab=64)
    inp = make_inputs(cfg, seed=6)
    ref_o, ref_l = oracle_attention(inp)
    for splits in (1, 2):
        out, lse = run_attention(sv, inp, num_splits=splits)
        check_attention(out, lse, ref_o, ref_l, label=f"H={H} k={k} splits={splits}")


def test_fold_equals_single_token_decode(sv):
    """A verify row equals a plain one-token decode of the same query and
    bound (bit for bit at one split): folding tokens into heads is exact."""
    inp = make_inputs(small_config("c0", R=2, k=3, H=64, kv_lens=(200, 77)), seed=7)
    d = device_inputs(inp, DEV)
    out, lse = sv.mla_verify_decode(d["q"], d["kv"], d["block_table"], d["kv_bounds"], d["gate"], 4,
                                    inp["softmax_scale"], num_splits=1)
    k1 = 4
    bt1 = torch.repeat_interleave(d["block_table"], k1, dim=0).contiguous()
    # one-token requests have 64 query rows: keep them on the same (two-CTA)
    # form as the verify groups
    out1, lse1 = sv.mla_verify_decode(d["q"], d["kv"], bt1, d["kv_bounds"], d["gate"], 1,
                                      inp["softmax_scale"], num_splits=1, form=sv.FORM_TWO_CTA)
    torch.cuda.synchronize()
    assert torch.equal(out, out1)
    assert torch.equal(lse, lse1)


def test_bad_device_data_sets_status(sv):
    inp = make_inputs(_mid_config(), seed=8)
    d = device_inputs(inp, DEV)
    bt = d["block_table"].clone()
    bt[1, 2] = inp["num_pages"] + 5  # a needed page id outside the pool
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sv.mla_verify_decode(d["q"], d["kv"], bt, d["kv_bounds"], d["gate"], inp["k"] + 1,
                         inp["softmax_scale"], num_splits=2, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & sv.SV_DEV_BAD_PAGE
    kb = d["kv_bounds"].clone()
    kb[0] = 10 ** 6  # beyond max_pages * 64
    status.zero_()
    sv.mla_verify_decode(d["q"], d["kv"], d["block_table"], kb, d["gate"], inp["k"] + 1,
                         inp["softmax_scale"], num_splits=1, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & sv.SV_DEV_BAD_BOUND
    # the context is still healthy: a clean call matches the oracle
    ref_o, ref_l = oracle_attention(inp)
    out, lse = run_attention(sv, inp)
    check_attention(out, lse, ref_o, ref_l, label="after bad data")


def test_empty_batch(sv):
    z = torch.empty((0, 64, 512), dtype=torch.bfloat16, device=DEV)
    kv = torch.zeros((1, 64, 512), dtype=torch.bfloat16, device=DEV)
    bt = torch.zeros((0, 1), dtype=torch.int32, device=DEV)
    kb = torch.zeros((0,), dtype=torch.int32, device=DEV)
    out, lse = sv.mla_verify_decode(z, kv, bt, kb, z, 1, 0.1)
    assert out.shape == (0, 64, 512) and lse.shape == (0, 64)


def test_verify_step_object(sv):
    inp = inputs_for("c1")
    d = device_inputs(inp, DEV)
    step = sv.VerifyStep(DEV, inp["R"], inp["k"], inp["H"], inp["cfg"].vocab, inp["max_pages"])
    res = step(d["q"], d["kv"], d["block_table"], d["kv_bounds"], d["gate"], inp["softmax_scale"],
               d["logits"], d["draft_tokens"], d["kv_lens_in"])
    torch.cuda.synchronize()
    ref = oracle.ref_verify_step(inp)
    check_attention(res[0], res[1], ref["out"], ref["lse"], label="step")
    for g, key in zip(res[2:], ("argmax", "accepted", "next_tokens", "kv_lens_out")):
        assert np.array_equal(g.cpu().numpy(), ref[key])


# ----------------------------------------------------------------- KV append
def _append_case(seed=10):
    cfg = small_config("c2", R=5, k=4, H=8, kv_lens=(64, 65, 700, 130, 5), kv_len_range=None,
                       shuffled=True, vocab=64)
    inp = make_inputs(cfg, seed=seed)
    k1 = inp["k"] + 1
    rng = np.random.default_rng(seed)
    from workloads import f32_to_bf16_bits
    kv_new = f32_to_bf16_bits(rng.standard_normal((inp["T"], 512), dtype=np.float32))
    pos = np.concatenate([np.arange(L - k1, L) for L in inp["kv_lens_in"]]).astype(np.int32)
    pos[3] = -1  # one token not written
    return inp, kv_new, pos


def test_kv_append_bit_exact(sv):
    inp, kv_new, pos = _append_case()
    k1 = inp["k"] + 1
    ref_pool = oracle.ref_kv_append(inp["kv_bits"], inp["block_table"], pos, kv_new, k1)
    d = device_inputs(inp, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sv.mla_kv_append(bf16_tensor(kv_new, DEV), i32(pos, DEV), d["block_table"], d["kv"], k1, status=status)
    torch.cuda.synchronize()
    got = d["kv"].view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, ref_pool)
    assert int(status.item()) == 0


def test_kv_append_then_attention(sv):
    """Append the verify rows, then attend: equals the oracle on the appended pool."""
    inp, kv_new, pos = _append_case(seed=11)
    k1 = inp["k"] + 1
    pool = oracle.ref_kv_append(inp["kv_bits"], inp["block_table"], pos, kv_new, k1)
    ref_o, ref_l = oracle.ref_verify_attention(inp["q_bits"], pool, inp["block_table"], inp["kv_bounds"],
                                               inp["gate_bits"], k1, inp["softmax_scale"])
    d = device_inputs(inp, DEV)
    sv.mla_kv_append(bf16_tensor(kv_new, DEV), i32(pos, DEV), d["block_table"], d["kv"], k1)
    out, lse = sv.mla_verify_decode(d["q"], d["kv"], d["block_table"], d["kv_bounds"], d["gate"], k1,
                                    inp["softmax_scale"])
    torch.cuda.synchronize()
    check_attention(out, lse, ref_o, ref_l, label="append+attention")


def test_kv_append_bad_data(sv):
    inp, kv_new, pos = _append_case(seed=12)
    k1 = inp["k"] + 1
    d = device_inputs(inp, DEV)
    before = d["kv"].clone()
    bad = pos.copy()
    bad[0] = inp["max_pages"] * 64 + 5  # past the block table
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sv.mla_kv_append(bf16_tensor(kv_new, DEV), i32(bad, DEV), d["block_table"], d["kv"], k1, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & sv.SV_DEV_BAD_BOUND
    # the bad token wrote nothing; the others match the oracle
    bad[0] = -1
    ref_pool = oracle.ref_kv_append(before.view(torch.int16).cpu().numpy().view(np.uint16),
                                    inp["block_table"], bad, kv_new, k1)
    assert np.array_equal(d["kv"].view(torch.int16).cpu().numpy().view(np.uint16), ref_pool)


# ----------------------------------------------------------------- balanced split plan
@pytest.mark.parametrize("lens", [(70, 4000, 333, 64, 1500), (5000,), (64, 65, 63, 4, 700, 2000, 129)])
def test_balanced_plan_matches_oracle(sv, lens):
    """Requests of very different lengths cut into pieces by the device-side plan."""
    cfg = small_config("c2", R=len(lens), k=3, H=32, kv_lens=lens, kv_len_range=None, shuffled=True,
                       vocab=64)
    inp = make_inputs(cfg, seed=21)
    ref_o, ref_l = oracle_attention(inp)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = run_attention(sv, inp, num_splits=sv.SV_SPLITS_BALANCED, status=status)
    assert int(status.item()) == 0
    check_attention(out, lse, ref_o, ref_l, label=f"balanced {lens}")


def test_balanced_plan_zero_bounds_and_nan_slack(sv):
    inp = make_inputs(_mid_config(kv_lens=(70, 2000, 333)), seed=22)
    k1 = inp["k"] + 1
    bounds = inp["kv_bounds"].copy()
    bounds[0] = 0
    bounds[k1:2 * k1] = 0  # the long request fully masked: one empty piece
    kv = inp["kv_bits"].copy()
    bt = inp["block_table"]
    for r in range(inp["R"]):
        L = int(inp["kv_lens_in"][r])
        last = int(bt[r, (L - 1) // 64])
        kv[last, L % 64 if L % 64 else 64:] = 0x7FC0
    ref_o, ref_l = oracle_attention(inp, bounds=bounds, kv_bits=kv)
    out, lse = run_attention(sv, inp, num_splits=sv.SV_SPLITS_BALANCED, bounds=bounds, kv_bits=kv)
    check_attention(out, lse, ref_o, ref_l, label="balanced zero bounds + nan slack")


@pytest.mark.parametrize("H,k,lens", [(96, 1, (300, 129, 3000)), (1, 0, (65, 1, 640)), (8, 19, (500, 64)),
                                      (3, 40, (700, 4200))])
def test_balanced_plan_head_shapes(sv, H, k, lens):
    cfg = small_config("c0", R=len(lens), k=k, H=H, kv_lens=lens, shuffled=True, vocab=64)
    inp = make_inputs(cfg, seed=23)
    ref_o, ref_l = oracle_attention(inp)
    out, lse = run_attention(sv, inp, num_splits=sv.SV_SPLITS_BALANCED)
    check_attention(out, lse, ref_o, ref_l, label=f"balanced H={H} k={k}")


@pytest.mark.parametrize("S", [1, 4, 5, 8, 9, 13, 21, 40])
def test_combine_split_counts(sv, S):
    """Every split-count bucket of the merge kernel (the first 4 / 8 / 12
    splits loaded with the weights, later ones in rounds), with uneven and
    empty ranges."""
    cfg = small_config("c0", R=2, k=3, H=16, kv_lens=(150, 260))
    inp = make_inputs(cfg, seed=20 + S)
    edges = []
    for L in (150, 260):
        cuts = sorted(np.random.default_rng(S + L).integers(0, L + 1, size=S - 1).tolist())
        edges.append([0] + cuts + [L])
    po, pl = oracle.ref_attention_partials(inp["q_bits"], inp["kv_bits"], inp["block_table"], inp["kv_bounds"], 4,
                                           inp["softmax_scale"], edges)
    ref_o, ref_l = oracle.ref_lse_combine(po, pl, inp["gate_bits"])
    out, lse = sv.mla_lse_combine(torch.from_numpy(po.astype(np.float32)).to(DEV),
                                  torch.from_numpy(pl.astype(np.float32)).to(DEV), bf16_tensor(inp["gate_bits"], DEV))
    torch.cuda.synchronize()
    check_attention(out, lse, ref_o, ref_l, label=f"combine S={S}")


def test_combine_ignores_values_of_empty_splits(sv):
    """A split with lse = -inf has weight 0; whatever its o holds (NaN here)
    must not reach the output (0 * NaN would poison the row)."""
    cfg = small_config("c0", R=2, k=3, H=16, kv_lens=(150, 260))
    inp = make_inputs(cfg, seed=9)
    edges = [[0, 150, 150, 150], [0, 0, 200, 260]]
    po, pl = oracle.ref_attention_partials(inp["q_bits"], inp["kv_bits"], inp["block_table"], inp["kv_bounds"], 4,
                                           inp["softmax_scale"], edges)
    ref_o, ref_l = oracle.ref_lse_combine(po, pl, inp["gate_bits"])
    po_nan = po.copy()
    po_nan[~np.isfinite(pl)] = np.nan
    out, lse = sv.mla_lse_combine(torch.from_numpy(po_nan.astype(np.float32)).to(DEV),
                                  torch.from_numpy(pl.astype(np.float32)).to(DEV), bf16_tensor(inp["gate_bits"], DEV))
    torch.cuda.synchronize()
    check_attention(out, lse, ref_o, ref_l, label="combine with NaN in empty splits")
