"""GPU parity of the head-wise gate and of the W_UV value up-projection
against the float64 oracle (C ABI calls)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import bf16_tensor, check_attention, device_inputs, to_f64
from workloads import f32_to_bf16_bits, make_inputs, small_config

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
WUV_REL_L2 = 5e-3   # bf16 output rounding (~2^-9 relative) after an fp32 sum of 512 products
WUV_MAX_REL = 2e-2  # per element, relative to the row's largest |v|


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verify_mla_gb300 as m
    m.load_library()
    return m


def _headwise(sv, inp, splits):
    g_head = np.ascontiguousarray(inp["gate_bits"][:, :, 0])
    d = device_inputs(inp, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = sv.mla_verify_decode(d["q"], d["kv"], d["block_table"], d["kv_bounds"], bf16_tensor(g_head, DEV),
                                    inp["k"] + 1, inp["softmax_scale"], num_splits=splits, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_o, ref_l = oracle.ref_verify_attention(inp["q_bits"], inp["kv_bits"], inp["block_table"], inp["kv_bounds"],
                                               g_head, inp["k"] + 1, inp["softmax_scale"])
    return out, lse, ref_o, ref_l


@pytest.mark.parametrize("splits", [1, 3, -1])
def test_headwise_gate(sv, splits):
    cfg = small_config("c2", R=3, k=4, H=64, kv_lens=(70, 700, 333), kv_len_range=None, shuffled=True, vocab=64)
    inp = make_inputs(cfg, seed=40)
    out, lse, ref_o, ref_l = _headwise(sv, inp, splits)
    check_attention(out, lse, ref_o, ref_l, label=f"head-wise gate, splits={splits}")


def test_headwise_gate_h96(sv):
    cfg = small_config("c0", R=2, k=1, H=96, kv_lens=(300, 1100), shuffled=True, vocab=64)
    inp = make_inputs(cfg, seed=41)
    for splits in (1, 2, -1):
        out, lse, ref_o, ref_l = _headwise(sv, inp, splits)
        check_attention(out, lse, ref_o, ref_l, label=f"H=96 head-wise, splits={splits}")


def _check_wuv(got, ref, label):
    g = to_f64(got)
    assert not np.any(np.isnan(g)), label
    rel = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30)
    assert rel <= WUV_REL_L2, f"{label}: rel-L2 {rel:.3e}"
    scale = np.max(np.abs(ref), axis=-1, keepdims=True) + 1e-30
    mx = np.max(np.abs(g - ref) / scale)
    assert mx <= WUV_MAX_REL, f"{label}: max rel {mx:.3e}"


@pytest.mark.parametrize("T,H,V", [(8, 64, 128), (160, 64, 128), (200, 3, 256), (1, 96, 32), (129, 2, 64), (40, 5, 96)])
def test_wuv_projection(sv, T, H, V):
    rng = np.random.default_rng(T * 1000 + H + V)
    x = f32_to_bf16_bits(rng.standard_normal((T, H, 512), dtype=np.float32))
    w = f32_to_bf16_bits((rng.standard_normal((H, V, 512), dtype=np.float32) / np.float32(16.0)))
    got = sv.mla_wuv_project(bf16_tensor(x, DEV), bf16_tensor(w, DEV))
    torch.cuda.synchronize()
    _check_wuv(got, oracle.ref_wuv_project(x, w), f"wuv T={T} H={H} V={V}")


def test_attention_then_wuv(sv):
    """The f4 chain: gated attention with a head-wise gate, merge, W_UV."""
    inp = make_inputs("c1", seed=3)
    H = inp["H"]
    g_head = np.ascontiguousarray(inp["gate_bits"][:, :, 0])
    rng = np.random.default_rng(5)
    w = f32_to_bf16_bits(rng.standard_normal((H, 128, 512), dtype=np.float32) / np.float32(16.0))
    d = device_inputs(inp, DEV)
    out, lse = sv.mla_verify_decode(d["q"], d["kv"], d["block_table"], d["kv_bounds"], bf16_tensor(g_head, DEV),
                                    inp["k"] + 1, inp["softmax_scale"])
    v = sv.mla_wuv_project(out, bf16_tensor(w, DEV))
    torch.cuda.synchronize()
    ref_o, _ = oracle.ref_verify_attention(inp["q_bits"], inp["kv_bits"], inp["block_table"], inp["kv_bounds"],
                                           g_head, inp["k"] + 1, inp["softmax_scale"])
    _check_wuv(v, oracle.ref_wuv_project(ref_o, w), "attention -> W_UV")
