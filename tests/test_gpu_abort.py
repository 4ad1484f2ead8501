"""The bounded waits of the attention kernel, made to run out on purpose.

Every wait of the attention kernel on an mbarrier phase gives up after a
limit (about two seconds in the library): the CTA then sets SV_DEV_TIMEOUT
in the status word, stops its pipeline, drains the copies and MMAs it
started, frees its TMEM and returns, so that a stalled pipeline becomes a
reported error instead of a hang or a silently wrong result (the guards of
"TensorRT-LLM PR #18166: Kimi K3 DSpark speculative decoding under Helix CP"
reject what they cannot serve loudly).  The test entry point
sv_test_mla_verify_decode_wait_limit lowers that limit per call.  Here it
is 0 (a wait gives up unless its phase has already completed), so the first
wait of the CTA for a copy in flight runs out, on every
kernel instance (bf16 and fp8 KV, two-CTA and stacked forms, one and two
score issuers) and with the split merge and the balanced plan behind it; and
a few microseconds on a larger batch, so that CTAs give up at different
points of their pipelines.  After each such call the device is still usable
and the next call, with the usual limit, matches the float64 oracle.  The
per-head W_UV projection kernel gets the same treatment.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_util import bf16_tensor, check_attention, device_inputs, to_f64
from workloads import f32_to_bf16_bits, fp8_kv_pool, make_inputs, small_config

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SV_DEV_TIMEOUT = 0x4
USUAL_LIMIT_NS = 2_000_000_000


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verify_mla_gb300 as m
    lib = m.load_library()
    f = lib.sv_test_mla_verify_decode_wait_limit
    c = ctypes
    f.argtypes = [c.c_void_p, c.c_void_p, c.c_int, c.c_float, c.c_int, c.c_int, c.c_void_p, c.c_int, c.c_int,
                  c.c_int, c.c_void_p, c.c_void_p, c.c_int, c.c_int, c.c_float, c.c_int, c.c_int, c.c_void_p,
                  c.c_size_t, c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p, c.c_uint64]
    f.restype = c.c_int
    g = lib.sv_test_mla_wuv_project_wait_limit
    g.argtypes = [c.c_void_p, c.c_void_p, c.c_int, c.c_int, c.c_int, c.c_void_p, c.c_void_p, c.c_void_p,
                  c.c_uint64]
    g.restype = c.c_int
    return m


def _call(sv, inp, fp8, splits, form, wait_ns):
    """One call of the test entry point; returns (out, lse, status word)."""
    d = device_inputs(inp, DEV)
    if fp8:
        codes, scale = fp8_kv_pool(inp)
        kv = torch.from_numpy(codes).to(DEV)
    else:
        kv, scale = d["kv"], 1.0
    R, k1, H, T = inp["R"], inp["k"] + 1, inp["H"], inp["T"]
    max_pages = inp["block_table"].shape[1]
    ws_bytes = sv.attention_workspace_bytes(T, H, splits)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=DEV)
    out = torch.full((T, H, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((T, H), float("nan"), dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    rc = sv.load_library().sv_test_mla_verify_decode_wait_limit(
        d["q"].data_ptr(), kv.data_ptr(), int(fp8), float(scale), int(inp["num_pages"]), 64,
        d["block_table"].data_ptr(), R, k1, max_pages, d["kv_bounds"].data_ptr(), d["gate"].data_ptr(), 512, H,
        float(inp["softmax_scale"]), splits, form, ws.data_ptr() if ws_bytes else None, ws_bytes, out.data_ptr(),
        lse.data_ptr(), status.data_ptr(), torch.cuda.current_stream().cuda_stream, wait_ns)
    assert rc == 0, rc
    torch.cuda.synchronize()  # raises if the context was lost
    return out, lse, int(status.item())


def _oracle(inp, fp8):
    kv = inp["kv_bits"]
    if fp8:
        codes, scale = fp8_kv_pool(inp)
        kv = oracle.e4m3_bits_to_f64(codes) * scale
    return oracle.ref_verify_attention(inp["q_bits"], kv, inp["block_table"], inp["kv_bounds"], inp["gate_bits"],
                                       inp["k"] + 1, inp["softmax_scale"])


# (num_splits, form): one split fused, two uniform splits and the merge, the
# balanced plan (two score issuers and the epilogue helpers), each form
_MODES = [(1, 1), (2, 1), (-1, 1), (1, 2), (2, 2)]


@pytest.mark.parametrize("fp8", [0, 1])
@pytest.mark.parametrize("splits,form", _MODES)
def test_wait_runs_out_then_next_call_is_exact(sv, fp8, splits, form):
    inp = make_inputs("c0", seed=5)
    _, _, st = _call(sv, inp, fp8, splits, form, wait_ns=0)
    assert st & SV_DEV_TIMEOUT, f"status {st:#x}: no wait ran out"
    assert st & ~SV_DEV_TIMEOUT == 0, f"status {st:#x}"
    out, lse, st = _call(sv, inp, fp8, splits, form, wait_ns=USUAL_LIMIT_NS)
    assert st == 0, f"status {st:#x}"
    ref_o, ref_l = _oracle(inp, fp8)
    check_attention(out, lse, ref_o, ref_l, label=f"after abort fp8={fp8} splits={splits} form={form}")


@pytest.mark.parametrize("limit_ns", [2_000, 20_000])
def test_waits_give_up_mid_pipeline_on_a_wave_batch(sv, limit_ns):
    """30 requests in the wave split mode (180 CTAs, the whole requests and
    the split pieces, the merge over the split rows): with a limit of a few
    microseconds some CTAs finish and others give up at different points of
    their pipelines.  Whatever each did, the call returns, the status word
    holds no other flag, and the next call is exact."""
    rng = np.random.default_rng(31)
    lens = tuple(int(x) for x in rng.integers(300, 1500, size=30))
    cfg = small_config("c2", R=30, k=4, H=64, kv_lens=lens, kv_len_range=None, shuffled=True, vocab=64)
    inp = make_inputs(cfg, seed=31)
    assert sv.num_splits_for(inp["R"], 5, 64, inp["max_pages"]) == sv.SV_SPLITS_WAVE
    _, _, st = _call(sv, inp, 0, sv.SV_SPLITS_WAVE, 0, wait_ns=limit_ns)
    assert st & ~SV_DEV_TIMEOUT == 0, f"status {st:#x}"
    out, lse, st = _call(sv, inp, 0, sv.SV_SPLITS_WAVE, 0, wait_ns=USUAL_LIMIT_NS)
    assert st == 0, f"status {st:#x}"
    ref_o, ref_l = _oracle(inp, 0)
    check_attention(out, lse, ref_o, ref_l, label=f"wave batch after a {limit_ns} ns limit")


@pytest.mark.parametrize("T,H,V", [(160, 4, 128), (40, 3, 256)])
def test_wuv_wait_runs_out_then_next_call_is_exact(sv, T, H, V):
    """The W_UV projection: with a zero limit every CTA's first wait for a
    copy gives up; the kernel writes no output row (the NaN fill stays) and
    returns; the next call is exact."""
    rng = np.random.default_rng(T + H + V)
    x = f32_to_bf16_bits(rng.standard_normal((T, H, 512), dtype=np.float32))
    w = f32_to_bf16_bits(rng.standard_normal((H, V, 512), dtype=np.float32) / np.float32(16.0))
    xd, wd = bf16_tensor(x, DEV), bf16_tensor(w, DEV)
    f = sv.load_library().sv_test_mla_wuv_project_wait_limit

    def call(limit):
        out = torch.full((T, H, V), float("nan"), dtype=torch.bfloat16, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        rc = f(xd.data_ptr(), wd.data_ptr(), T, H, V, out.data_ptr(), status.data_ptr(),
               torch.cuda.current_stream().cuda_stream, limit)
        assert rc == 0, rc
        torch.cuda.synchronize()
        return out, int(status.item())

    out, st = call(0)
    assert st == SV_DEV_TIMEOUT, f"status {st:#x}"
    assert torch.isnan(out.float()).all()  # every CTA gave up and wrote nothing
    out, st = call(USUAL_LIMIT_NS)
    assert st == 0, f"status {st:#x}"
    ref = oracle.ref_wuv_project(x, w)
    g = to_f64(out)
    rel = np.linalg.norm(g - ref) / np.linalg.norm(ref)
    assert rel <= 5e-3, f"W_UV after abort: rel-L2 {rel:.3e}"  # bf16 output rounding, as the W_UV parity
