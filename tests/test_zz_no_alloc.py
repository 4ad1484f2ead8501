"""The allocation-free greedy verify entry point.

spec_verify_greedy_noalloc exists for callers that cannot allocate device
memory when they verify (an engine whose KV-cache pool already holds nearly
all of HBM, or a plugin whose host framework owns the allocator), so they
cannot hand spec_verify_greedy a workspace.  It keeps its scratch in a static
device array instead.  This test calls it through the C ABI twice in a row
(the array keeps the previous call's contents) and checks that every output
equals the workspace entry point's output on the same inputs.  The file name
makes pytest collect it after every other test file.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _lib():
    from speculative_decoding_verify_mla_gb300 import load_library
    lib = load_library()
    f = lib.spec_verify_greedy_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return lib


def _noalloc(lib, logits, drafts, kv_in, k):
    T, V = logits.shape
    R = kv_in.shape[0]
    outs = [torch.full((n,), -7, dtype=torch.int32, device=DEV) for n in (T, R, R, R)]
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.spec_verify_greedy_noalloc(logits.data_ptr(), T, V, R, k,
                                        drafts.data_ptr() if k > 0 else None, kv_in.data_ptr(),
                                        *[o.data_ptr() for o in outs], stream)
    assert rc == 0, rc
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in outs]


@pytest.mark.parametrize("name", ["c0", "c1", "c2"])
def test_noalloc_matches_workspace_entry_point(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verify_mla_gb300 as sv
    from workloads import make_inputs
    lib = _lib()
    inp = make_inputs(name, seed=11)
    k = inp["k"]
    logits = torch.from_numpy(inp["logits"]).to(DEV)
    drafts = torch.from_numpy(np.ascontiguousarray(inp["draft_tokens"])).to(DEV)
    kv_in = torch.from_numpy(inp["kv_lens_in"]).to(DEV)
    ref = [t.cpu().numpy() for t in sv.spec_verify_greedy(logits, drafts, kv_in, k)]
    for _ in range(2):  # two calls in a row share (and reuse) the static scratch
        got = _noalloc(lib, logits, drafts, kv_in, k)
        for g, r in zip(got, ref):
            assert np.array_equal(g, r)


def test_noalloc_rejects_problems_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verify_mla_gb300 as sv
    lib = _lib()
    T, V = 1 << 16, 1 << 20  # 12 bytes of scratch per token: more than 512 KiB
    assert sv.greedy_workspace_bytes(T, V) > 512 * 1024
    rc = lib.spec_verify_greedy_noalloc(4096, T, V, T, 0, None, 4096, 4096, 4096, 4096, 4096, None)
    assert rc == 4  # SV_ERR_WORKSPACE, nothing enqueued
