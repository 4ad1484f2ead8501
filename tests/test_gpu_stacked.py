"""GPU parity of the stacked attention form (requests of at most 64 query
rows on one CTA that holds both latent halves) against the float64 oracle,
with the form chosen per call (forced on, forced off, automatic) on the same
inputs, under uniform splits and the balanced plan (C ABI calls)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import bf16_tensor, check_attention, device_inputs, i32, to_f64
from workloads import make_inputs, small_config

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verify_mla_gb300 as m
    m.load_library()
    return m


def form_of(sv, on):
    """The per-call kernel form: stacked (True), two CTAs (False), or the
    given SV_FORM_* value."""
    if isinstance(on, bool):
        return sv.FORM_STACKED if on else sv.FORM_TWO_CTA
    return on


def _attention(sv, inp, splits, bounds=None, kv_bits=None, gate_bits=None, form=0):
    d = device_inputs(inp, DEV)
    kv = d["kv"] if kv_bits is None else bf16_tensor(kv_bits, DEV)
    kb = d["kv_bounds"] if bounds is None else i32(bounds, DEV)
    gate = d["gate"] if gate_bits is None else bf16_tensor(gate_bits, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = sv.mla_verify_decode(d["q"], kv, d["block_table"], kb, gate, inp["k"] + 1, inp["softmax_scale"],
                                    num_splits=splits, status=status, form=form)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out, lse


def _oracle(inp, bounds=None, kv_bits=None, gate_bits=None):
    return oracle.ref_verify_attention(inp["q_bits"], inp["kv_bits"] if kv_bits is None else kv_bits,
                                       inp["block_table"], inp["kv_bounds"] if bounds is None else bounds,
                                       inp["gate_bits"] if gate_bits is None else gate_bits, inp["k"] + 1,
                                       inp["softmax_scale"])


# M = H (k+1) <= 64 in every case: plain decode at H = 64 (ragged lengths,
# a 1-position request (k = 0), a long one that takes the two-score-issuer instance),
# partial 64-row tiles (M = 32, 63, 1) and M = 64 exactly.
SHAPES = [(64, 0, (1100, 1500, 64, 1, 700)), (8, 3, (64, 100)), (16, 3, (333, 65, 4)), (1, 0, (65, 1, 640)),
          (32, 1, (129, 2000)), (64, 0, (5000,)), (3, 20, (700, 300))]


@pytest.mark.parametrize("H,k,lens", SHAPES)
@pytest.mark.parametrize("on", [True, False])
def test_stacked_matches_oracle(sv, H, k, lens, on):
    cfg = small_config("c0", R=len(lens), k=k, H=H, kv_lens=lens, shuffled=True, vocab=64)
    inp = make_inputs(cfg, seed=11)
    ref_o, ref_l = _oracle(inp)
    for splits in (1, 2, 5, 0, sv.SV_SPLITS_BALANCED):
        out, lse = _attention(sv, inp, splits, form=form_of(sv, on))
        check_attention(out, lse, ref_o, ref_l, label=f"stacked={on} H={H} k={k} splits={splits}")


def test_stacked_zero_bounds_nan_slack_headwise_gate(sv):
    """Fully masked tokens and requests, NaN pool slack past each request's
    last row, and the head-wise gate, through the stacked form."""
    cfg = small_config("c0", R=3, k=3, H=16, kv_lens=(70, 700, 333), shuffled=True, vocab=64)
    inp = make_inputs(cfg, seed=12)
    k1 = inp["k"] + 1
    bounds = inp["kv_bounds"].copy()
    bounds[0] = 0
    bounds[k1:2 * k1] = 0
    kv = inp["kv_bits"].copy()
    for r in range(inp["R"]):
        L = int(inp["kv_lens_in"][r])
        kv[int(inp["block_table"][r, (L - 1) // 64]), L % 64 if L % 64 else 64:] = 0x7FC0
    ref_o, ref_l = _oracle(inp, bounds=bounds, kv_bits=kv)
    g_head = np.ascontiguousarray(inp["gate_bits"][:, :, 0])
    ref_oh, ref_lh = _oracle(inp, bounds=bounds, kv_bits=kv, gate_bits=g_head)
    for splits in (1, 4, sv.SV_SPLITS_BALANCED):
        out, lse = _attention(sv, inp, splits, bounds=bounds, kv_bits=kv, form=sv.FORM_STACKED)
        check_attention(out, lse, ref_o, ref_l, label=f"zero bounds + nan slack, splits={splits}")
        out, lse = _attention(sv, inp, splits, bounds=bounds, kv_bits=kv, gate_bits=g_head, form=sv.FORM_STACKED)
        check_attention(out, lse, ref_oh, ref_lh, label=f"head-wise gate, splits={splits}")


def test_stacked_partials_layout(sv):
    """Split partials of the stacked form follow the documented workspace
    layout (both latent halves of every row written)."""
    cfg = small_config("c0", R=3, k=0, H=64, kv_lens=(70, 700, 333), shuffled=True, vocab=64)
    inp = make_inputs(cfg, seed=13)
    S = 3
    d = device_inputs(inp, DEV)
    T, H = inp["T"], inp["H"]
    ws = torch.empty(sv.attention_workspace_bytes(T, H, S), dtype=torch.uint8, device=DEV)
    sv.mla_verify_decode(d["q"], d["kv"], d["block_table"], d["kv_bounds"], d["gate"], 1,
                         inp["softmax_scale"], num_splits=S, workspace=ws, form=sv.FORM_STACKED)
    torch.cuda.synchronize()
    n_o = S * T * H * 512
    part_o = ws[:2 * n_o].view(torch.bfloat16).view(S, T, H, 512)
    part_lse = ws[2 * n_o:2 * n_o + 4 * S * T * H].view(torch.float32).view(S, T, H)
    edges = []
    for r in range(inp["R"]):
        n_r = -(-int(inp["kv_bounds"][r]) // 64)
        edges.append([64 * ((s * n_r) // S) for s in range(S + 1)])
    po, pl = oracle.ref_attention_partials(inp["q_bits"], inp["kv_bits"], inp["block_table"], inp["kv_bounds"],
                                           1, inp["softmax_scale"], edges)
    gl = to_f64(part_lse)
    assert np.array_equal(np.isfinite(gl), np.isfinite(pl))
    fin = np.isfinite(pl)
    assert np.max(np.abs(gl[fin] - pl[fin])) <= 1e-3
    go = to_f64(part_o)
    assert np.linalg.norm(go - po) / np.linalg.norm(po) <= 1e-2
    assert np.all(go[~fin] == 0.0)


def test_stacked_equals_two_cta_form(sv):
    """Both forms compute the same scores and softmax (LSE bit for bit); the
    stacked P V also runs MMAs whose A block is zero, which the tensor core's
    fp32 accumulation does not always leave bit-identical, so the outputs
    agree to rounding: far tighter than the oracle tolerance."""
    cfg = small_config("c0", R=4, k=0, H=64, kv_lens=(1100, 64, 1, 700), shuffled=True, vocab=64)
    inp = make_inputs(cfg, seed=14)
    o1, l1 = _attention(sv, inp, 1, form=sv.FORM_STACKED)
    o2, l2 = _attention(sv, inp, 1, form=sv.FORM_TWO_CTA)
    assert torch.equal(l1, l2)
    a, b = o1.double(), o2.double()
    rel = float(torch.linalg.norm(a - b) / torch.linalg.norm(b))
    mx = float((a - b).abs().max())
    assert rel <= 2e-3 and mx <= 4e-3, f"rel-L2 {rel:.3e}, max abs {mx:.3e}"


def test_auto_splits_count_one_cta_per_unit(sv):
    """The automatic split count of the stacked form fills the SMs with one
    CTA per (request, split)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    s_auto = sv.num_splits_for(64, 1, 64, 24, sv.FORM_AUTO)
    s_short = sv.num_splits_for(2, 4, 8, 2, sv.FORM_AUTO)  # 1-2 tile units keep the two-CTA form
    s_off = sv.num_splits_for(64, 1, 64, 24, sv.FORM_TWO_CTA)
    assert s_auto == max(1, min(sms // 64, 12))
    assert s_off == max(1, min(sms // 128, 12))
    assert s_short == 1


def test_stacked_balanced_plan_c3(sv):
    """The C = 64 plain-decode batch (64 requests x 16-24 KV tiles) in the
    stacked form under the balanced plan (pieces of ceil(sum n_r / SMs)
    tiles, one CTA each, partials merged per request), and the two-CTA form
    under the same plan, against the oracle over every token and head."""
    inp = make_inputs("c3", seed=0)
    ref_o, ref_l = _oracle(inp)
    for form in (sv.FORM_STACKED, sv.FORM_TWO_CTA):
        out, lse = _attention(sv, inp, sv.SV_SPLITS_BALANCED, form=form)
        check_attention(out, lse, ref_o, ref_l, label=f"c3 balanced plan, form={form}")


def test_stacked_balanced_plan_long_context(sv):
    """Plain decode at long context (16 requests of 8K-32K positions, k = 0,
    H = 64: 64 rows per request, 10% zero bounds): the automatic choice is
    the balanced plan in the stacked form; every token and head against the
    oracle."""
    inp = make_inputs(small_config("c4", k=0), seed=0)
    assert sv.num_splits_for(inp["R"], 1, 64, inp["max_pages"]) == sv.SV_SPLITS_BALANCED
    ref_o, ref_l = _oracle(inp)
    out, lse = _attention(sv, inp, 0)
    check_attention(out, lse, ref_o, ref_l, label="long-context plain decode, balanced plan, stacked")
