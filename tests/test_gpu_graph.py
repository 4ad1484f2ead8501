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
