"""ctypes binding of libspecverify.so: argument marshalling only.

Every step of the verify path runs in the library's CUDA kernels; this module
checks torch tensor dtypes/devices/shapes, allocates outputs and workspaces
with torch (the library itself never allocates), and passes raw device
pointers plus the current CUDA stream.  There is no fallback: if the library
is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB_PATH

_c_int = ctypes.c_int
_c_size = ctypes.c_size_t
_c_float = ctypes.c_float
_c_void_p = ctypes.c_void_p

SV_LATENT_DIM = 512
SV_PAGE_SIZE = 64
SV_MAX_SPLITS = 64
SV_SPLITS_BALANCED = -1
SV_SPLITS_WAVE = -2
# kernel form of the attention call (SV_FORM_*), chosen per call
FORM_AUTO, FORM_TWO_CTA, FORM_STACKED = 0, 1, 2
SV_DEV_BAD_PAGE = 0x1
SV_DEV_BAD_BOUND = 0x2
SV_DEV_TIMEOUT = 0x4

EXPORTED_SYMBOLS = (
    "sv_status_string",
    "sv_mla_verify_num_splits",
    "sv_mla_verify_workspace_bytes",
    "mla_verify_decode",
    "mla_lse_combine",
    "sv_greedy_workspace_bytes",
    "spec_verify_greedy",
    "mla_kv_append",
    "sv_sampled_workspace_bytes",
    "spec_verify_sampled",
    "mla_verify_decode_gated",
    "mla_wuv_project",
    "mla_verify_decode_kv8",
)

_lib = None
_lock = threading.Lock()


class SpecVerifyError(RuntimeError):
    def __init__(self, func: str, code: int):
        self.code = code
        super().__init__(f"{func} failed: {status_string(code)} (code {code})")


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load (once) the compiled library; raises if it has not been built.
    The environment variable SPECVERIFY_LIBRARY names another build of it
    (e.g. the index-checking debug build) to load instead."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or os.environ.get("SPECVERIFY_LIBRARY") or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it first "
                "(python -m speculative_decoding_verify_mla_gb300.build)")
        lib = ctypes.CDLL(path)
        lib.sv_status_string.argtypes = [_c_int]
        lib.sv_status_string.restype = ctypes.c_char_p
        lib.sv_mla_verify_num_splits.argtypes = [_c_int, _c_int, _c_int, _c_int, _c_int]
        lib.sv_mla_verify_num_splits.restype = _c_int
        lib.sv_mla_verify_workspace_bytes.argtypes = [_c_int, _c_int, _c_int]
        lib.sv_mla_verify_workspace_bytes.restype = _c_size
        lib.mla_verify_decode.argtypes = [
            _c_void_p, _c_void_p, _c_int, _c_int, _c_void_p, _c_int, _c_int, _c_int, _c_void_p,
            _c_void_p, _c_int, _c_float, _c_int, _c_void_p, _c_size, _c_void_p, _c_void_p,
            _c_void_p, _c_void_p]
        lib.mla_verify_decode.restype = _c_int
        lib.mla_lse_combine.argtypes = [_c_void_p, _c_void_p, _c_int, _c_int, _c_int, _c_void_p,
                                        _c_void_p, _c_void_p, _c_void_p]
        lib.mla_lse_combine.restype = _c_int
        lib.sv_greedy_workspace_bytes.argtypes = [_c_int, _c_int]
        lib.sv_greedy_workspace_bytes.restype = _c_size
        lib.spec_verify_greedy.argtypes = [
            _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
            _c_void_p, _c_void_p, _c_void_p, _c_size, _c_void_p]
        lib.spec_verify_greedy.restype = _c_int
        lib.mla_kv_append.argtypes = [_c_void_p, _c_void_p, _c_void_p, _c_int, _c_int, _c_int,
                                      _c_void_p, _c_int, _c_int, _c_void_p, _c_void_p]
        lib.mla_kv_append.restype = _c_int
        lib.sv_sampled_workspace_bytes.argtypes = [_c_int, _c_int, _c_int]
        lib.sv_sampled_workspace_bytes.restype = _c_size
        lib.spec_verify_sampled.argtypes = [
            _c_void_p, _c_int, _c_int, _c_int, _c_float, _c_void_p, _c_void_p, _c_void_p,
            _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_size, _c_void_p]
        lib.spec_verify_sampled.restype = _c_int
        lib.mla_verify_decode_gated.argtypes = [
            _c_void_p, _c_void_p, _c_int, _c_int, _c_void_p, _c_int, _c_int, _c_int, _c_void_p,
            _c_void_p, _c_int, _c_int, _c_float, _c_int, _c_int, _c_void_p, _c_size, _c_void_p,
            _c_void_p, _c_void_p, _c_void_p]
        lib.mla_verify_decode_gated.restype = _c_int
        lib.mla_wuv_project.argtypes = [_c_void_p, _c_void_p, _c_int, _c_int, _c_int, _c_void_p,
                                        _c_void_p, _c_void_p]
        lib.mla_wuv_project.restype = _c_int
        lib.mla_verify_decode_kv8.argtypes = [
            _c_void_p, _c_void_p, _c_float, _c_int, _c_int, _c_void_p, _c_int, _c_int, _c_int,
            _c_void_p, _c_void_p, _c_int, _c_int, _c_float, _c_int, _c_int, _c_void_p, _c_size,
            _c_void_p, _c_void_p, _c_void_p, _c_void_p]
        lib.mla_verify_decode_kv8.restype = _c_int
        _lib = lib
        return lib


def status_string(code: int) -> str:
    return load_library().sv_status_string(int(code)).decode()


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _check_status(func: str, code: int):
    if code != 0:
        raise SpecVerifyError(func, code)


def num_splits_for(R: int, q_per_req: int, H: int, max_pages_per_req: int, form: int = FORM_AUTO) -> int:
    """The split count num_splits = 0 resolves to for this form."""
    s = int(load_library().sv_mla_verify_num_splits(R, q_per_req, H, max_pages_per_req, int(form)))
    if s == 0:
        raise ValueError(f"unknown attention form {form}")
    return s


def attention_workspace_bytes(T: int, H: int, num_splits: int) -> int:
    return int(load_library().sv_mla_verify_workspace_bytes(T, H, num_splits))


def greedy_workspace_bytes(T: int, V: int) -> int:
    return int(load_library().sv_greedy_workspace_bytes(T, V))


def mla_verify_decode(q_latent: torch.Tensor, kv_pages: torch.Tensor, block_table: torch.Tensor,
                      kv_bounds: torch.Tensor, gate: torch.Tensor, q_per_req: int,
                      softmax_scale: float, num_splits: int = 0,
                      workspace: torch.Tensor | None = None, out: torch.Tensor | None = None,
                      lse: torch.Tensor | None = None, status: torch.Tensor | None = None,
                      kv_scale: float | None = None, form: int = FORM_AUTO):
    """Gated NoPE MLA verify attention.  Shapes: q_latent [T, H, 512] bf16,
    gate [T, H, 512] or [T, H] bf16, kv_pages [P, 64, 512] bf16 (or uint8 E4M3
    codes with kv_scale given), block_table [R, max_pages] int32, kv_bounds [T]
    int32.  ``form`` picks the kernel form (FORM_AUTO, FORM_TWO_CTA or
    FORM_STACKED) for this call.  Returns (out [T, H, 512] bf16, lse [T, H]
    fp32)."""
    lib = load_library()
    _check(q_latent.dim() == 3 and q_latent.shape[2] == SV_LATENT_DIM, "q_latent must be [T, H, 512]")
    T, H, _ = q_latent.shape
    dev = q_latent.device
    _check(dev.type == "cuda", "tensors must live on a CUDA device")
    kv8 = kv_scale is not None
    for name, t, dt in (("q_latent", q_latent, torch.bfloat16),
                        ("kv_pages", kv_pages, torch.uint8 if kv8 else torch.bfloat16),
                        ("gate", gate, torch.bfloat16), ("block_table", block_table, torch.int32),
                        ("kv_bounds", kv_bounds, torch.int32)):
        _check(t.dtype == dt, f"{name} must be {dt}")
        _check(t.device == dev, f"{name} must be on {dev}")
        _check(t.is_contiguous(), f"{name} must be contiguous")
    _check(kv_pages.dim() == 3 and kv_pages.shape[2] == SV_LATENT_DIM, "kv_pages must be [P, page, 512]")
    _check(tuple(gate.shape) in ((T, H, SV_LATENT_DIM), (T, H)),
           "gate must be [T, H, 512] (elementwise) or [T, H] (head-wise)")
    gate_dim = SV_LATENT_DIM if gate.dim() == 3 else 1
    _check(block_table.dim() == 2, "block_table must be [R, max_pages]")
    R, max_pages = block_table.shape
    _check(T == R * q_per_req, "T must equal R * q_per_req")
    _check(tuple(kv_bounds.shape) == (T,), "kv_bounds must be [T]")
    if num_splits == 0:
        num_splits = num_splits_for(R, q_per_req, H, max_pages, form)
    if out is None:
        out = torch.empty((T, H, SV_LATENT_DIM), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    ws_bytes = attention_workspace_bytes(T, H, num_splits)
    if ws_bytes > 0 and (workspace is None or workspace.numel() * workspace.element_size() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    ws_size = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if kv8:
        code = lib.mla_verify_decode_kv8(
            _ptr(q_latent), _ptr(kv_pages), float(kv_scale), int(kv_pages.shape[0]),
            int(kv_pages.shape[1]), _ptr(block_table), R, q_per_req, max_pages, _ptr(kv_bounds),
            _ptr(gate), gate_dim, H, float(softmax_scale), int(num_splits), int(form), _ptr(workspace),
            ws_size, _ptr(out), _ptr(lse), _ptr(status), _stream(dev))
    else:
        code = lib.mla_verify_decode_gated(
            _ptr(q_latent), _ptr(kv_pages), int(kv_pages.shape[0]), int(kv_pages.shape[1]),
            _ptr(block_table), R, q_per_req, max_pages, _ptr(kv_bounds), _ptr(gate), gate_dim, H,
            float(softmax_scale), int(num_splits), int(form), _ptr(workspace), ws_size, _ptr(out),
            _ptr(lse), _ptr(status), _stream(dev))
    _check_status("mla_verify_decode", code)
    return out, lse


def mla_lse_combine(part_o: torch.Tensor, part_lse: torch.Tensor, gate: torch.Tensor,
                    out: torch.Tensor | None = None, lse: torch.Tensor | None = None):
    """LSE merge of split partials + sigmoid gate.  part_o [S, T, H, 512] fp32,
    part_lse [S, T, H] fp32, gate [T, H, 512] bf16 -> (out bf16, lse fp32)."""
    lib = load_library()
    _check(part_o.dim() == 4 and part_o.shape[3] == SV_LATENT_DIM, "part_o must be [S, T, H, 512]")
    S, T, H, _ = part_o.shape
    dev = part_o.device
    _check(part_o.dtype == torch.float32 and part_lse.dtype == torch.float32, "partials must be fp32")
    _check(tuple(part_lse.shape) == (S, T, H), "part_lse must be [S, T, H]")
    _check(gate.dtype == torch.bfloat16 and tuple(gate.shape) == (T, H, SV_LATENT_DIM), "gate must be [T, H, 512] bf16")
    for t in (part_o, part_lse, gate):
        _check(t.is_contiguous() and t.device == dev, "tensors must be contiguous and on one device")
    if out is None:
        out = torch.empty((T, H, SV_LATENT_DIM), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    code = lib.mla_lse_combine(_ptr(part_o), _ptr(part_lse), S, T, H, _ptr(gate), _ptr(out),
                               _ptr(lse), _stream(dev))
    _check_status("mla_lse_combine", code)
    return out, lse


_greedy_ws: dict = {}


def greedy_workspace(device: torch.device, T: int, V: int) -> torch.Tensor:
    """A zero-filled greedy workspace, cached per device and size (each call
    leaves it zero-filled again, so it is reused as is)."""
    need = greedy_workspace_bytes(T, V)
    key = (str(device), need)
    ws = _greedy_ws.get(key)
    if ws is None:
        ws = torch.zeros(need, dtype=torch.uint8, device=device)
        _greedy_ws[key] = ws
    return ws


def spec_verify_greedy(logits: torch.Tensor, draft_tokens: torch.Tensor, kv_lens_in: torch.Tensor,
                       k: int, workspace: torch.Tensor | None = None, argmax_ids=None,
                       accepted=None, next_tokens=None, kv_lens_out=None):
    """Greedy verify.  logits [R*(k+1), V] fp32, draft_tokens [R, k] int32,
    kv_lens_in [R] int32 -> (argmax [T], accepted [R], next_tokens [R],
    kv_lens_out [R]), all int32."""
    lib = load_library()
    _check(logits.dim() == 2 and logits.dtype == torch.float32, "logits must be [T, V] fp32")
    T, V = logits.shape
    dev = logits.device
    R = kv_lens_in.shape[0]
    _check(T == R * (k + 1), "T must equal R * (k + 1)")
    _check(kv_lens_in.dtype == torch.int32 and kv_lens_in.is_contiguous(), "kv_lens_in must be int32")
    _check(draft_tokens.dtype == torch.int32 and draft_tokens.is_contiguous(), "draft_tokens must be int32")
    _check(tuple(draft_tokens.shape) == (R, k), "draft_tokens must be [R, k]")
    _check(logits.is_contiguous(), "logits must be contiguous")
    if workspace is None:
        workspace = greedy_workspace(dev, T, V)
    outs = []
    for t, n in ((argmax_ids, T), (accepted, R), (next_tokens, R), (kv_lens_out, R)):
        outs.append(torch.empty(n, dtype=torch.int32, device=dev) if t is None else t)
    code = lib.spec_verify_greedy(
        _ptr(logits), T, V, R, k, _ptr(draft_tokens) if k > 0 else None, _ptr(kv_lens_in),
        *[_ptr(o) for o in outs], _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(dev))
    _check_status("spec_verify_greedy", code)
    return tuple(outs)


def mla_kv_append(kv_new: torch.Tensor, positions: torch.Tensor, block_table: torch.Tensor,
                  kv_pages: torch.Tensor, q_per_req: int, status: torch.Tensor | None = None):
    """Write kv_new [T, 512] bf16 into kv_pages [P, 64, 512] (in place) at the
    tokens' positions [T] int32 (-1 = skip) through block_table [R, max_pages]."""
    lib = load_library()
    _check(kv_new.dim() == 2 and kv_new.shape[1] == SV_LATENT_DIM, "kv_new must be [T, 512]")
    T = kv_new.shape[0]
    R, max_pages = block_table.shape
    _check(T == R * q_per_req, "T must equal R * q_per_req")
    dev = kv_new.device
    for name, t, dt in (("kv_new", kv_new, torch.bfloat16), ("kv_pages", kv_pages, torch.bfloat16),
                        ("positions", positions, torch.int32), ("block_table", block_table, torch.int32)):
        _check(t.dtype == dt and t.device == dev and t.is_contiguous(), f"{name}: {dt}, contiguous, on {dev}")
    _check(tuple(positions.shape) == (T,), "positions must be [T]")
    code = lib.mla_kv_append(_ptr(kv_new), _ptr(positions), _ptr(block_table), R, q_per_req,
                             max_pages, _ptr(kv_pages), int(kv_pages.shape[0]),
                             int(kv_pages.shape[1]), _ptr(status), _stream(dev))
    _check_status("mla_kv_append", code)
    return kv_pages


def sampled_workspace_bytes(R: int, k: int, V: int) -> int:
    return int(load_library().sv_sampled_workspace_bytes(R, k, V))


_sampled_ws: dict = {}


def sampled_workspace(device, R: int, k: int, V: int) -> torch.Tensor:
    """A zero-filled workspace for spec_verify_sampled, cached per device and
    size (the kernels leave its counters zero after every call)."""
    key = (str(device), sampled_workspace_bytes(R, k, V))
    ws = _sampled_ws.get(key)
    if ws is None:
        ws = torch.zeros(key[1], dtype=torch.uint8, device=device)
        _sampled_ws[key] = ws
    return ws


def spec_verify_sampled(logits: torch.Tensor, draft_tokens: torch.Tensor, draft_probs: torch.Tensor,
                        uniforms: torch.Tensor, kv_lens_in: torch.Tensor, k: int,
                        temperature: float = 1.0, workspace: torch.Tensor | None = None,
                        accepted: torch.Tensor | None = None, next_tokens: torch.Tensor | None = None,
                        kv_lens_out: torch.Tensor | None = None):
    """Rejection-sampling verification.  logits [R*(k+1), V] fp32, draft_tokens
    [R, k] int32, draft_probs [R, k, V] fp32, uniforms [R, k+1] fp32, kv_lens_in
    [R] int32.  Returns (accepted, next_tokens, kv_lens_out), each [R] int32."""
    lib = load_library()
    _check(logits.dim() == 2, "logits must be [T, V]")
    T, V = logits.shape
    R = kv_lens_in.shape[0]
    _check(T == R * (k + 1), "T must equal R * (k + 1)")
    dev = logits.device
    _check(dev.type == "cuda", "tensors must live on a CUDA device")
    checks = [("logits", logits, torch.float32), ("uniforms", uniforms, torch.float32),
              ("kv_lens_in", kv_lens_in, torch.int32)]
    if k > 0:
        checks += [("draft_tokens", draft_tokens, torch.int32), ("draft_probs", draft_probs, torch.float32)]
        _check(tuple(draft_tokens.shape) == (R, k), "draft_tokens must be [R, k]")
        _check(tuple(draft_probs.shape) == (R, k, V), "draft_probs must be [R, k, V]")
    for name, t, dt in checks:
        _check(t.dtype == dt and t.device == dev and t.is_contiguous(), f"{name}: {dt}, contiguous, on {dev}")
    _check(tuple(uniforms.shape) == (R, k + 1), "uniforms must be [R, k+1]")
    if workspace is None:
        workspace = sampled_workspace(dev, R, k, V)
    outs = []
    for o in (accepted, next_tokens, kv_lens_out):
        outs.append(torch.empty(R, dtype=torch.int32, device=dev) if o is None else o)
    code = lib.spec_verify_sampled(
        _ptr(logits), R, k, V, float(temperature), _ptr(draft_tokens) if k > 0 else None,
        _ptr(draft_probs) if k > 0 else None, _ptr(uniforms), _ptr(kv_lens_in),
        _ptr(outs[0]), _ptr(outs[1]), _ptr(outs[2]), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(dev))
    _check_status("spec_verify_sampled", code)
    return tuple(outs)


def mla_wuv_project(x: torch.Tensor, w_uv: torch.Tensor, out_v: torch.Tensor | None = None,
                    status: torch.Tensor | None = None) -> torch.Tensor:
    """Per-head value up-projection: x [T, H, 512] bf16, w_uv [H, v_dim, 512]
    bf16 -> out_v [T, H, v_dim] bf16."""
    lib = load_library()
    _check(x.dim() == 3 and x.shape[2] == SV_LATENT_DIM, "x must be [T, H, 512]")
    T, H, _ = x.shape
    _check(w_uv.dim() == 3 and w_uv.shape[0] == H and w_uv.shape[2] == SV_LATENT_DIM,
           "w_uv must be [H, v_dim, 512]")
    v_dim = int(w_uv.shape[1])
    dev = x.device
    for name, t in (("x", x), ("w_uv", w_uv)):
        _check(t.dtype == torch.bfloat16 and t.device == dev and t.is_contiguous(),
               f"{name}: bf16, contiguous, on {dev}")
    if out_v is None:
        out_v = torch.empty((T, H, v_dim), dtype=torch.bfloat16, device=dev)
    code = lib.mla_wuv_project(_ptr(x), _ptr(w_uv), T, H, v_dim, _ptr(out_v), _ptr(status), _stream(dev))
    _check_status("mla_wuv_project", code)
    return out_v
