"""The boundary's own attention entry point, mla_verify_decode, called
through ctypes with raw device pointers (no Python binding in between) on the
tiny and the C=32 verify batches, against the float64 oracle.  The per-token
kv_bounds interface it implements is the one of "TensorRT-LLM PR #18166: Kimi
K3 DSpark speculative decoding under Helix CP" (first commit message)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_attention, device_inputs
from workloads import make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verify_mla_gb300 import load_library
    return load_library()


@pytest.mark.parametrize("name,splits", [("c0", 0), ("c0", 2), ("c2", 0), ("c2", 3), ("c2", -1)])
def test_literal_entry_point_matches_oracle(lib, name, splits):
    inp = make_inputs(name, seed=0)
    d = device_inputs(inp, DEV)
    R, k1, H, T = inp["R"], inp["k"] + 1, inp["H"], inp["T"]
    max_pages = inp["block_table"].shape[1]
    S = splits if splits != 0 else lib.sv_mla_verify_num_splits(R, k1, H, max_pages, 0)
    ws_bytes = lib.sv_mla_verify_workspace_bytes(T, H, S)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=DEV)
    out = torch.full((T, H, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((T, H), float("nan"), dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.mla_verify_decode(d["q"].data_ptr(), d["kv"].data_ptr(), int(inp["num_pages"]), 64,
                               d["block_table"].data_ptr(), R, k1, max_pages, d["kv_bounds"].data_ptr(),
                               d["gate"].data_ptr(), H, ctypes.c_float(inp["softmax_scale"]), splits,
                               ws.data_ptr() if ws_bytes else None, ws_bytes, out.data_ptr(), lse.data_ptr(),
                               status.data_ptr(), stream)
    assert rc == 0, rc
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_o, ref_l = oracle.ref_verify_attention(inp["q_bits"], inp["kv_bits"], inp["block_table"],
                                               inp["kv_bounds"], inp["gate_bits"], k1, inp["softmax_scale"])
    check_attention(out, lse, ref_o, ref_l, label=f"mla_verify_decode {name} splits={splits}")


def test_literal_entry_point_zero_bounds(lib):
    """Fully masked tokens through the literal entry point give (-inf, 0)."""
    inp = make_inputs("c0", seed=3)
    d = device_inputs(inp, DEV)
    bounds = inp["kv_bounds"].copy()
    bounds[[0, 5]] = 0
    kb = torch.from_numpy(bounds).to(DEV)
    R, k1, H, T = inp["R"], inp["k"] + 1, inp["H"], inp["T"]
    out = torch.full((T, H, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((T, H), float("nan"), dtype=torch.float32, device=DEV)
    rc = lib.mla_verify_decode(d["q"].data_ptr(), d["kv"].data_ptr(), int(inp["num_pages"]), 64,
                               d["block_table"].data_ptr(), R, k1, inp["block_table"].shape[1], kb.data_ptr(),
                               d["gate"].data_ptr(), H, ctypes.c_float(inp["softmax_scale"]), 1, None, 0,
                               out.data_ptr(), lse.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
    assert rc == 0, rc
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.ref_verify_attention(inp["q_bits"], inp["kv_bits"], inp["block_table"], bounds,
                                               inp["gate_bits"], k1, inp["softmax_scale"])
    check_attention(out, lse, ref_o, ref_l, label="mla_verify_decode zero bounds")
    assert np.all(lse.cpu().numpy()[[0, 5]] == -np.inf)
