"""Helpers for the GPU parity tests: move generated inputs to the device and
compare device outputs with the float64 oracle."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances for the attention output against the unrounded float64 oracle
# (bf16 inputs, bf16 P in the P.V product, fp32 accumulation, bf16 output):
OUT_REL_L2 = 1e-2     # ||out - ref||_2 / ||ref||_2 over the whole output
OUT_MAX_ABS = 2e-2    # max |out - ref|
LSE_MAX_ABS = 1e-3    # max |lse - ref| over finite entries


def bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def i32(x: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).to(device)


def device_inputs(inp: dict, device="cuda:0") -> dict:
    return dict(
        q=bf16_tensor(inp["q_bits"], device),
        kv=bf16_tensor(inp["kv_bits"], device),
        gate=bf16_tensor(inp["gate_bits"], device),
        block_table=i32(inp["block_table"], device),
        kv_bounds=i32(inp["kv_bounds"], device),
        logits=torch.from_numpy(np.ascontiguousarray(inp["logits"])).to(device),
        draft_tokens=i32(inp["draft_tokens"].reshape(inp["R"], inp["k"]), device),
        kv_lens_in=i32(inp["kv_lens_in"], device),
    )


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_attention(out: torch.Tensor, lse: torch.Tensor, ref_out: np.ndarray, ref_lse: np.ndarray,
                    rows=None, label=""):
    o = to_f64(out)
    l = to_f64(lse)
    if rows is not None:
        o, l = o[rows], l[rows]
    assert not np.any(np.isnan(o)), f"{label}: NaN in out"
    assert not np.any(np.isnan(l)), f"{label}: NaN in lse"
    ref_fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(l), ref_fin), f"{label}: -inf pattern of lse differs"
    assert np.all(l[~ref_fin] == -np.inf), f"{label}: masked rows must have lse = -inf"
    assert np.all(o[~ref_fin] == 0.0), f"{label}: masked rows must have out = 0"
    if ref_fin.any():
        lse_err = np.max(np.abs(l[ref_fin] - ref_lse[ref_fin]))
        assert lse_err <= LSE_MAX_ABS, f"{label}: lse max abs err {lse_err:.3e}"
    diff = o - ref_out
    denom = np.linalg.norm(ref_out)
    rel = np.linalg.norm(diff) / denom if denom > 0 else np.linalg.norm(diff)
    mx = np.max(np.abs(diff)) if diff.size else 0.0
    assert rel <= OUT_REL_L2, f"{label}: out rel-L2 {rel:.3e}"
    assert mx <= OUT_MAX_ABS, f"{label}: out max abs {mx:.3e}"
    return rel, mx
