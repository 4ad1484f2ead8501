"""The allocation-free greedy verify entry point.

spec_verify_greedy_noalloc exists for callers that cannot allocate device
memory when they verify (an engine whose KV-cache pool already holds nearly
all of HBM, or a plugin whose host framework owns the allocator), so they
cannot hand spec_verify_greedy a workspace.  It keeps its scratch in a static
device array instead, shared by every call and keeping the last call's
contents.  These tests call it through the C ABI and check that every output
equals the workspace entry point's output on the same inputs: twice in a row
on one batch, on batches of different sizes one after another (a large batch,
then a small one, then the large one again, so a partly used array is reused),
and on the largest batch the array holds.  The file name makes pytest collect
it after every other test file.
"""
import ctypes

import numpy as np
import pytest
import torch

DEV = "cuda:0"
SCRATCH_BYTES = 512 * 1024


def _lib():
    from speculative_decoding_verify_mla_gb300 import build as B
    B.build()
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


def _device_batch(inp):
    logits = torch.from_numpy(inp["logits"]).to(DEV)
    drafts = torch.from_numpy(np.ascontiguousarray(inp["draft_tokens"])).to(DEV)
    kv_in = torch.from_numpy(inp["kv_lens_in"]).to(DEV)
    return logits, drafts, kv_in


def _check_against_workspace_entry(lib, logits, drafts, kv_in, k):
    import speculative_decoding_verify_mla_gb300 as sv
    ref = [t.cpu().numpy() for t in sv.spec_verify_greedy(logits, drafts, kv_in, k)]
    got = _noalloc(lib, logits, drafts, kv_in, k)
    for g, r in zip(got, ref):
        assert np.array_equal(g, r)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["c0", "c1", "c2"])
def test_noalloc_matches_workspace_entry_point(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from workloads import make_inputs
    lib = _lib()
    inp = make_inputs(name, seed=11)
    logits, drafts, kv_in = _device_batch(inp)
    for _ in range(2):  # two calls in a row share (and reuse) the static scratch
        _check_against_workspace_entry(lib, logits, drafts, kv_in, inp["k"])


@pytest.mark.gpu
def test_noalloc_large_small_large():
    """A large batch, then a small one, then the large one again on one
    stream: each call clears only the part of the array it uses, so the
    small call runs on a partly used array and the large one after it on an
    array whose tail the small call never touched."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from workloads import make_inputs
    lib = _lib()
    big, small = make_inputs("c2", seed=12), make_inputs("c0", seed=13)
    for inp in (big, small, big):
        _check_against_workspace_entry(lib, *_device_batch(inp), inp["k"])


@pytest.mark.gpu
def test_noalloc_largest_batch_that_fits():
    """The largest T whose scratch (256 + 8 T bytes) fits in 512 KiB, with
    planted maxima and ties, against the workspace entry point."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verify_mla_gb300 as sv
    lib = _lib()
    k = 1
    T = (SCRATCH_BYTES - 256) // 8
    T -= T % (k + 1)
    R, V = T // (k + 1), 12
    assert sv.greedy_workspace_bytes(T, V) <= SCRATCH_BYTES < sv.greedy_workspace_bytes(T + 2, V)
    rng = np.random.default_rng(14)
    x = rng.integers(-3, 4, size=(T, V)).astype(np.float32)  # many ties
    drafts = rng.integers(0, V, size=(R, k)).astype(np.int32)
    kv_in = rng.integers(10, 1000, size=R).astype(np.int32)
    _check_against_workspace_entry(lib, torch.from_numpy(x).to(DEV), torch.from_numpy(drafts).to(DEV),
                                   torch.from_numpy(kv_in).to(DEV), k)


@pytest.mark.gpu
def test_noalloc_rejects_bad_calls_without_device_pointers():
    """Argument errors come back on the host; every device pointer here is
    NULL, so no call below can reach device memory whatever the check order."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _lib()
    f = lib.spec_verify_greedy_noalloc
    T, V = 1 << 16, 1 << 20  # 8 bytes of scratch per token: more than 512 KiB
    assert f(None, T, V, T, 0, None, None, None, None, None, None, None) == 1   # SV_ERR_NULL
    assert f(None, 7, V, 2, 3, None, None, None, None, None, None, None) == 2   # T != R (k + 1)
    assert f(None, 0, V, 0, 3, None, None, None, None, None, None, None) == 0   # nothing to do


def test_noalloc_size_limit_is_checked_first_on_the_host():
    """Without a GPU: an oversize problem is rejected with SV_ERR_WORKSPACE
    before any CUDA call (a CUDA call here, with no device, would fail with
    SV_ERR_DEVICE), and the other argument checks come before the size
    check.  The made-up addresses are never dereferenced: there is no device,
    and the test is skipped where there is one."""
    if torch.cuda.is_available():
        pytest.skip("host-only check (runs where no GPU is present)")
    lib = _lib()
    f = lib.spec_verify_greedy_noalloc
    T, V = 1 << 16, 1 << 20
    a = 1 << 12
    assert f(a, T, V, T, 0, None, a, a, a, a, a, None) == 4           # SV_ERR_WORKSPACE
    assert f(a + 2, T, V, T, 0, None, a, a, a, a, a, None) == 3       # logits alignment first
    assert f(a, T, V, T, 0, None, a, None, a, a, a, None) == 1        # null output first
    assert f(a, 8, 64, 2, 3, a, a, a, a, a, a, None) == 9             # fits: reaches CUDA, no device
