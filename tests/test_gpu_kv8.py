"""GPU parity of the fp8 (E4M3 + scale) latent KV variant against the float64
oracle over the dequantised pool (C ABI calls)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import bf16_tensor, check_attention, device_inputs, i32
from workloads import fp8_kv_pool, make_inputs, small_config

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verify_mla_gb300 as m
    m.load_library()
    return m


def _run(sv, inp, splits, gate=None, bounds=None, status=None, form=0):
    codes, scale = fp8_kv_pool(inp)
    d = device_inputs(inp, DEV)
    kv8 = torch.from_numpy(codes).to(DEV)
    g = d["gate"] if gate is None else bf16_tensor(gate, DEV)
    b = d["kv_bounds"] if bounds is None else i32(bounds, DEV)
    out, lse = sv.mla_verify_decode(d["q"], kv8, d["block_table"], b, g, inp["k"] + 1, inp["softmax_scale"],
                                    num_splits=splits, status=status, kv_scale=scale, form=form)
    torch.cuda.synchronize()
    deq = oracle.e4m3_bits_to_f64(codes) * scale
    ref_o, ref_l = oracle.ref_verify_attention(inp["q_bits"], deq, inp["block_table"],
                                               inp["kv_bounds"] if bounds is None else bounds,
                                               inp["gate_bits"] if gate is None else gate, inp["k"] + 1,
                                               inp["softmax_scale"])
    return out, lse, ref_o, ref_l


@pytest.mark.parametrize("name", ["c0", "c1", "c2", "c3"])
def test_kv8_configs(sv, name):
    inp = make_inputs(name, seed=0)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse, ref_o, ref_l = _run(sv, inp, 0, status=status)
    assert int(status.item()) == 0
    check_attention(out, lse, ref_o, ref_l, label=f"kv8 {name}")


@pytest.mark.parametrize("splits", [1, 3, 7, -1])
def test_kv8_splits_and_plan(sv, splits):
    cfg = small_config("c2", R=4, k=4, H=64, kv_lens=(70, 1900, 333, 64), kv_len_range=None, shuffled=True,
                       vocab=64)
    inp = make_inputs(cfg, seed=50)
    out, lse, ref_o, ref_l = _run(sv, inp, splits)
    check_attention(out, lse, ref_o, ref_l, label=f"kv8 splits={splits}")


@pytest.mark.parametrize("splits", [2, -1])
def test_kv8_stacked_splits_and_plan(sv, splits):
    """The fp8 stacked form (M = 64 rows per request) under uniform splits and
    the balanced plan, ragged contexts."""
    cfg = small_config("c3", R=5, k=0, H=64, kv_lens=(70, 1900, 333, 64, 1200), kv_len_range=None, shuffled=True,
                       vocab=64)
    inp = make_inputs(cfg, seed=51)
    out, lse, ref_o, ref_l = _run(sv, inp, splits, form=sv.FORM_STACKED)
    check_attention(out, lse, ref_o, ref_l, label=f"kv8 stacked splits={splits}")


@pytest.mark.parametrize("mode", ["always", "off"])
@pytest.mark.parametrize("H,k,lens", [(64, 0, (1100, 64, 4, 700)), (16, 3, (333, 65, 4)), (8, 3, (64, 100))])
def test_kv8_stacked_form(sv, mode, H, k, lens):
    """Requests of <= 64 query rows over an fp8 pool, with the stacked form
    (one CTA holding both latent halves) forced on and off; zero bounds and
    the head-wise gate included."""
    cfg = small_config("c0", R=len(lens), k=k, H=H, kv_lens=lens, shuffled=True, vocab=64)
    inp = make_inputs(cfg, seed=52)
    bounds = inp["kv_bounds"].copy()
    bounds[0] = 0
    g_head = np.ascontiguousarray(inp["gate_bits"][:, :, 0])
    form = sv.FORM_STACKED if mode == "always" else sv.FORM_TWO_CTA
    for splits in (1, 3, 0):
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        out, lse, ref_o, ref_l = _run(sv, inp, splits, bounds=bounds, status=status, form=form)
        assert int(status.item()) == 0
        check_attention(out, lse, ref_o, ref_l, label=f"kv8 stacked={mode} H={H} k={k} splits={splits}")
    out, lse, ref_o, ref_l = _run(sv, inp, 2, gate=g_head, bounds=bounds, form=form)
    check_attention(out, lse, ref_o, ref_l, label=f"kv8 stacked={mode} head gate")


def test_kv8_zero_bounds_headwise_h96(sv):
    cfg = small_config("c0", R=3, k=1, H=96, kv_lens=(300, 129, 800), shuffled=True, vocab=64)
    inp = make_inputs(cfg, seed=51)
    bounds = inp["kv_bounds"].copy()
    bounds[0] = 0
    bounds[2:4] = 0
    g_head = np.ascontiguousarray(inp["gate_bits"][:, :, 0])
    for splits in (1, 2, -1):
        out, lse, ref_o, ref_l = _run(sv, inp, splits, gate=g_head, bounds=bounds)
        check_attention(out, lse, ref_o, ref_l, label=f"kv8 H=96 head gate zero bounds splits={splits}")


def test_kv8_equals_bf16_on_exact_pool(sv):
    """A bf16 pool holding exactly the fp8 values (codes x scale with a power-
    of-two scale) gives the same result through both variants."""
    inp = make_inputs(small_config("c0", R=2, k=3, H=16, kv_lens=(200, 77)), seed=52)
    codes, _ = fp8_kv_pool(inp)
    scale = 0.0078125  # 2^-7: codes x scale are exact in bf16
    deq = (oracle.e4m3_bits_to_f64(codes) * scale).astype(np.float32)
    deq_bits = (np.ascontiguousarray(deq).view(np.uint32) >> 16).astype(np.uint16)
    d = device_inputs(inp, DEV)
    o8, l8 = sv.mla_verify_decode(d["q"], torch.from_numpy(codes).to(DEV), d["block_table"], d["kv_bounds"],
                                  d["gate"], 4, inp["softmax_scale"], num_splits=1, kv_scale=scale)
    o16, l16 = sv.mla_verify_decode(d["q"], bf16_tensor(deq_bits, DEV), d["block_table"], d["kv_bounds"],
                                    d["gate"], 4, inp["softmax_scale"], num_splits=1)
    torch.cuda.synchronize()
    assert torch.allclose(o8.float(), o16.float(), rtol=2e-2, atol=2e-3)
    fin = torch.isfinite(l16)
    assert torch.equal(torch.isfinite(l8), fin)
    assert torch.allclose(l8[fin], l16[fin], rtol=0, atol=1e-4)


def test_kv8_c4_full(sv):
    """The full-size long-context workload over the fp8 pool (balanced plan)
    against the oracle on every token and head; the oracle reads each
    request's dequantised pages only (decoded through the oracle's own table
    of all 256 codes)."""
    inp = make_inputs("c4", seed=0)
    codes, scale = fp8_kv_pool(inp)
    d = device_inputs(inp, DEV)
    kv8 = torch.from_numpy(codes).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = sv.mla_verify_decode(d["q"], kv8, d["block_table"], d["kv_bounds"], d["gate"], inp["k"] + 1,
                                    inp["softmax_scale"], status=status, kv_scale=scale)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    del kv8
    k1 = inp["k"] + 1
    T, H = inp["T"], inp["H"]
    ref_o = np.zeros((T, H, 512))
    ref_l = np.zeros((T, H))
    lut = oracle.e4m3_bits_to_f64(np.arange(256, dtype=np.uint8)) * scale
    for r in range(inp["R"]):
        toks = slice(r * k1, (r + 1) * k1)
        n_pages = -(-int(inp["kv_bounds"][toks].max()) // 64)
        pool = lut[codes[inp["block_table"][r, :max(n_pages, 1)]]]  # this request's pages, in order
        o_r, l_r = oracle.ref_verify_attention(inp["q_bits"][toks], pool, np.arange(max(n_pages, 1))[None, :],
                                               inp["kv_bounds"][toks], inp["gate_bits"][toks], k1,
                                               inp["softmax_scale"])
        ref_o[toks], ref_l[toks] = o_r, l_r
    check_attention(out, lse, ref_o, ref_l, label="kv8 c4 full")
