"""A seeded sweep of the attention over shapes and modes, against the
float64 oracle.

Every attention case draws a batch (1-12 requests, k = 0-9, H from 1 to 128, context
lengths from 1 to 2500 positions, shuffled block tables), sets about 10% of
the tokens' bounds to 0 (the (-inf, 0) rows of "TensorRT-LLM PR #18166: Kimi
K3 DSpark speculative decoding under Helix CP", zero-bound commit messages)
and fills the pool slack past each request's last position with NaN, then
runs the kernel under three (split mode, kernel form) choices drawn from
uniform splits, the balanced plan and the automatic choice, and the two-CTA,
stacked and automatic forms, with bf16 or fp8 KV and the elementwise or
head-wise gate.  Two more batches sit in the wave split mode's range.  The
greedy verify gets the same treatment over shapes and tie patterns, and
the paged KV append over batch shapes and skipped tokens.  The cases come
from fixed seeds, so a failure names a reproducible case.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import bf16_tensor, check_attention, device_inputs, i32
from workloads import fp8_kv_pool, make_inputs, small_config

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
NAN_BF16 = 0x7FC0
NAN_E4M3 = 0x7F


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verify_mla_gb300 as m
    m.load_library()
    return m


def _case(i):
    """Batch shape, seed and modes of sweep case i (deterministic)."""
    rng = np.random.default_rng(9000 + i)
    R = int(rng.integers(1, 13))
    k = int(rng.integers(0, 10))
    H = int(rng.choice([1, 3, 8, 16, 32, 64, 96, 128]))
    while H * (k + 1) * R > 6000:  # keeps the oracle to a second or two per case
        k = max(0, k // 2)
        R = max(1, R - 2)
    kind = rng.random(R)
    lens = np.where(kind < 0.15, rng.integers(1, 5, R),
                    np.where(kind < 0.3, 64 * rng.integers(1, 20, R), rng.integers(1, 2501, R)))
    lens = tuple(int(max(x, k + 1)) for x in lens)
    fp8 = bool(rng.random() < 0.4)
    head_gate = bool(rng.random() < 0.3)
    modes = [(0, 0)]
    choices = [(1, 1), (3, 1), (-1, 1), (1, 2), (3, 2), (-1, 2), (0, 1), (0, 2), (5, 0), (-1, 0)]
    for j in rng.choice(len(choices), size=2, replace=False):
        modes.append(choices[int(j)])
    return R, k, H, lens, fp8, head_gate, modes


def _slack(inp):
    """(page, first slack row) of every request whose last page is partial."""
    out = []
    for r in range(inp["R"]):
        L = int(inp["kv_lens_in"][r])
        if L % 64:
            out.append((int(inp["block_table"][r, (L - 1) // 64]), L % 64))
    return out


def _prepare(inp, seed):
    """Zero ~10% of the bounds and put NaN in the pool slack."""
    rng = np.random.default_rng(seed)
    bounds = inp["kv_bounds"].copy()
    bounds[rng.random(bounds.shape[0]) < 0.1] = 0
    kv = inp["kv_bits"].copy()
    for page, row in _slack(inp):
        kv[page, row:] = NAN_BF16
    return bounds, kv


def _run(sv, inp, bounds, kv_bits, fp8, gate_bits, splits, form):
    d = device_inputs(inp, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    if fp8:
        # the scale of the clean pool, then NaN codes in the slack
        codes, scale = fp8_kv_pool(inp)
        kv_ref = oracle.e4m3_bits_to_f64(codes) * scale
        codes = codes.copy()
        for page, row in _slack(inp):
            codes[page, row:] = NAN_E4M3
        kv = torch.from_numpy(codes).to(DEV)
    else:
        kv, scale, kv_ref = bf16_tensor(kv_bits, DEV), None, kv_bits
    out, lse = sv.mla_verify_decode(d["q"], kv, d["block_table"], i32(bounds, DEV), bf16_tensor(gate_bits, DEV),
                                    inp["k"] + 1, inp["softmax_scale"], num_splits=splits, status=status,
                                    kv_scale=scale, form=form)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out, lse, kv_ref


@pytest.mark.parametrize("i", range(64))
def test_sweep_case(sv, i):
    R, k, H, lens, fp8, head_gate, modes = _case(i)
    cfg = small_config("c0", R=R, k=k, H=H, kv_lens=lens, kv_len_range=None, shuffled=True, vocab=64)
    inp = make_inputs(cfg, seed=100 + i)
    bounds, kv_bits = _prepare(inp, 200 + i)
    gate = np.ascontiguousarray(inp["gate_bits"][:, :, 0]) if head_gate else inp["gate_bits"]
    ref = None
    for splits, form in modes:
        out, lse, kv_ref = _run(sv, inp, bounds, kv_bits, fp8, gate, splits, form)
        if ref is None:
            ref = oracle.ref_verify_attention(inp["q_bits"], kv_ref, inp["block_table"], bounds, gate, k + 1,
                                              inp["softmax_scale"])
        check_attention(out, lse, *ref, label=f"case {i} R={R} k={k} H={H} fp8={fp8} head_gate={head_gate} "
                                             f"splits={splits} form={form}")


@pytest.mark.parametrize("fp8", [False, True])
def test_sweep_wave_mode(sv, fp8):
    """A batch whose unsplit units fill the SMs between once and twice: the
    automatic choice is the wave split mode, run here with zero bounds and
    NaN slack."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rng = np.random.default_rng(77 + fp8)
    R = sms // 6 + 8  # 3 row tiles x 2 halves per request: between one and two waves
    lens = tuple(int(x) for x in rng.integers(260, 1800, size=R))
    cfg = small_config("c2", R=R, k=4, H=64, kv_lens=lens, kv_len_range=None, shuffled=True, vocab=64)
    inp = make_inputs(cfg, seed=300 + fp8)
    assert sv.num_splits_for(R, 5, 64, inp["max_pages"]) == sv.SV_SPLITS_WAVE
    bounds, kv_bits = _prepare(inp, 400 + fp8)
    out, lse, kv_ref = _run(sv, inp, bounds, kv_bits, fp8, inp["gate_bits"], sv.SV_SPLITS_WAVE, 0)
    ref = oracle.ref_verify_attention(inp["q_bits"], kv_ref, inp["block_table"], bounds, inp["gate_bits"], 5,
                                      inp["softmax_scale"])
    check_attention(out, lse, *ref, label=f"wave mode fp8={fp8}")


@pytest.mark.parametrize("i", range(32))
def test_sweep_greedy(sv, i):
    """Greedy verify on seeded shapes (1-40 requests, k = 0-12, V from 1 to
    200003, odd and even), logits drawn from a few integer levels so that
    the row maxima repeat (ties across threads, chunks and CTAs; signed
    zeros), drafts that follow the argmax chain for a random number of steps
    then differ: bit for bit against the oracle, twice in a row (the second
    call checks that the first left its workspace clean)."""
    rng = np.random.default_rng(5000 + i)
    R = int(rng.integers(1, 41))
    k = int(rng.integers(0, 13))
    V = int(rng.choice([1, 2, 3, 5, 64, 1000, 4097, 8192, 16385, 65536, 163840, 200003]))
    while R * (k + 1) * V > 20_000_000:
        R = max(1, R // 2)
    T = R * (k + 1)
    levels = np.array([-3.0, -0.0, 0.0, 1.5, 2.0], dtype=np.float32)
    x = levels[rng.integers(0, len(levels), size=(T, V))]
    a_ref = np.argmax(x, axis=1)  # numpy picks the first maximum (ties, and -0 == +0)
    drafts = np.zeros((R, k), dtype=np.int32)
    for r in range(R):
        n_match = int(rng.integers(0, k + 1))
        for j in range(k):
            a = int(a_ref[r * (k + 1) + j])
            drafts[r, j] = a if j < n_match else (a + 1 + int(rng.integers(0, max(1, V - 1)))) % V
    kv_in = rng.integers(k + 1, 5000, size=R).astype(np.int32)
    ref = oracle.ref_greedy_verify(x, drafts, kv_in, k)
    lt = torch.from_numpy(np.ascontiguousarray(x)).to(DEV)
    dt = torch.from_numpy(drafts).to(DEV)
    kt = torch.from_numpy(kv_in).to(DEV)
    ws = torch.zeros(sv.greedy_workspace_bytes(T, V), dtype=torch.uint8, device=DEV)
    for _ in range(2):
        got = [t.cpu().numpy() for t in sv.spec_verify_greedy(lt, dt, kt, k, workspace=ws)]
        for g, r in zip(got, ref):
            assert np.array_equal(g, np.asarray(r)), f"case {i}: R={R} k={k} V={V}"


@pytest.mark.parametrize("i", range(16))
def test_sweep_kv_append(sv, i):
    """The paged KV append on seeded batches (1-24 requests, k = 0-15,
    shuffled tables): the verify group's rows go to the positions just below
    each request's length (crossing page boundaries), about 10% of the tokens
    are skipped (-1); the pool must equal the oracle's bit for bit."""
    rng = np.random.default_rng(6000 + i)
    R = int(rng.integers(1, 25))
    k = int(rng.integers(0, 16))
    lens = tuple(int(x) for x in rng.integers(k + 1, 3000, size=R))
    cfg = small_config("c0", R=R, k=k, H=8, kv_lens=lens, kv_len_range=None, shuffled=True, vocab=64)
    inp = make_inputs(cfg, seed=6100 + i)
    k1 = k + 1
    pos = np.empty(R * k1, dtype=np.int32)
    for r in range(R):
        L = int(inp["kv_lens_in"][r])
        pos[r * k1:(r + 1) * k1] = np.arange(L - k1, L)
    pos[rng.random(pos.shape[0]) < 0.1] = -1
    kv_new = rng.integers(0, 1 << 16, size=(R * k1, 512)).astype(np.uint16)
    kv_new[(kv_new & 0x7F80) == 0x7F80] &= 0xBFFF  # no NaN / inf patterns among the random rows
    ref = oracle.ref_kv_append(inp["kv_bits"], inp["block_table"], pos, kv_new, k1)
    d = device_inputs(inp, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sv.mla_kv_append(bf16_tensor(kv_new, DEV), i32(pos, DEV), d["block_table"], d["kv"], k1, status=status)
    torch.cuda.synchronize()
    got = d["kv"].view(torch.int16).cpu().numpy().view(np.uint16)
    assert int(status.item()) == 0
    assert np.array_equal(got, ref), f"case {i}: R={R} k={k}"
