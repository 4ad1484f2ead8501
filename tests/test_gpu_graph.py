"""The verify step captured in a CUDA graph (the pages run verification inside
captured graphs): replays equal eager execution bit for bit, for the uniform
split path, the balanced plan (plan kernel + programmatic dependent launches)
and the side-stream greedy verify."""
import numpy as np
import pytest
import torch

from gpu_util import device_inputs
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


@pytest.mark.parametrize("name,splits", [("c1", 0), ("c2", 0), ("c2", -1), ("c4-small", -1)])
def test_graph_replay_equals_eager(sv, name, splits):
    if name == "c4-small":
        cfg = small_config("c4", R=4, kv_len_range=(4096, 9000), vocab=4096)
    else:
        cfg = name
    inp = make_inputs(cfg, seed=60)
    d = device_inputs(inp, DEV)
    V = inp["logits"].shape[1]
    step = sv.VerifyStep(DEV, inp["R"], inp["k"], inp["H"], V, inp["max_pages"], num_splits=splits)

    def run():
        return step(d["q"], d["kv"], d["block_table"], d["kv_bounds"], d["gate"], inp["softmax_scale"],
                    d["logits"], d["draft_tokens"], d["kv_lens_in"])

    run()
    torch.cuda.synchronize()
    eager = [t.clone() for t in run()]
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device=DEV)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            res = run()
    torch.cuda.synchronize()
    for _ in range(3):
        for t in res:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(res, eager):
            assert torch.equal(a, b)
    assert int(step.status.item()) == 0


def test_staged_inputs_one_copy(sv):
    """StagedInputs: one host-to-device copy brings every input; the step's
    results come back as one [3, R] block."""
    inp = make_inputs("c1", seed=61)
    d = device_inputs(inp, DEV)
    specs = {k: (tuple(d[k].shape), d[k].dtype) for k in ("q", "gate", "logits", "block_table", "kv_bounds",
                                                            "draft_tokens", "kv_lens_in")}
    st = sv.StagedInputs(DEV, specs)
    for k in specs:
        st.host[k].copy_(d[k].cpu())
    st.upload()
    torch.cuda.synchronize()
    for k in specs:
        assert torch.equal(st.dev[k], d[k])
        assert st.dev[k].data_ptr() % 256 == 0
    V = inp["logits"].shape[1]
    step = sv.VerifyStep(DEV, inp["R"], inp["k"], inp["H"], V, inp["max_pages"])
    res = step(st.dev["q"], d["kv"], st.dev["block_table"], st.dev["kv_bounds"], st.dev["gate"],
               inp["softmax_scale"], st.dev["logits"], st.dev["draft_tokens"], st.dev["kv_lens_in"])
    torch.cuda.synchronize()
    assert torch.equal(step.results[0], res[3]) and torch.equal(step.results[1], res[4])
    assert torch.equal(step.results[2], res[5])


def test_run_staged_equals_device_step(sv):
    inp = make_inputs("c2", seed=62)
    d = device_inputs(inp, DEV)
    V = inp["logits"].shape[1]
    step = sv.VerifyStep(DEV, inp["R"], inp["k"], inp["H"], V, inp["max_pages"])
    ref = [t.clone() for t in step(d["q"], d["kv"], d["block_table"], d["kv_bounds"], d["gate"],
                                   inp["softmax_scale"], d["logits"], d["draft_tokens"], d["kv_lens_in"])]
    torch.cuda.synchronize()
    att = sv.StagedInputs(DEV, {"q_latent": (tuple(d["q"].shape), d["q"].dtype),
                                "gate": (tuple(d["gate"].shape), d["gate"].dtype),
                                "block_table": (tuple(d["block_table"].shape), torch.int32),
                                "kv_bounds": (tuple(d["kv_bounds"].shape), torch.int32)})
    ver = sv.StagedInputs(DEV, {"logits": (tuple(d["logits"].shape), torch.float32),
                                "draft_tokens": (tuple(d["draft_tokens"].shape), torch.int32),
                                "kv_lens_in": (tuple(d["kv_lens_in"].shape), torch.int32)})
    for k, src in (("q_latent", "q"), ("gate", "gate"), ("block_table", "block_table"), ("kv_bounds", "kv_bounds")):
        att.host[k].copy_(d[src].cpu())
    for k in ("logits", "draft_tokens", "kv_lens_in"):
        ver.host[k].copy_(d[k].cpu())
    step.out.zero_()
    res = step.run_staged(att, ver, d["kv"], inp["softmax_scale"])
    torch.cuda.synchronize()
    assert torch.equal(step.out, ref[0]) and torch.equal(step.lse, ref[1])
    assert torch.equal(res[0], ref[3]) and torch.equal(res[1], ref[4]) and torch.equal(res[2], ref[5])
