"""The seeded input generator: determinism, shapes and structure (CPU only)."""
import numpy as np
import pytest

from workloads import CONFIGS, causal_bounds, make_inputs, small_config


def test_deterministic():
    a = make_inputs("c0", seed=0)
    b = make_inputs("c0", seed=0)
    for key in ("q_bits", "kv_bits", "gate_bits", "logits", "draft_tokens", "block_table", "kv_bounds"):
        assert np.array_equal(a[key], b[key]), key
    c = make_inputs("c0", seed=1)
    assert not np.array_equal(a["q_bits"], c["q_bits"])


def test_c0_shapes_and_bounds():
    inp = make_inputs("c0")
    assert inp["q_bits"].shape == (8, 8, 512) and inp["q_bits"].dtype == np.uint16
    assert inp["kv_bits"].shape == (1 + 2, 64, 512)
    assert list(inp["kv_lens_in"]) == [64, 100]
    assert list(inp["kv_bounds"]) == [61, 62, 63, 64, 97, 98, 99, 100]
    assert inp["logits"].shape == (8, 1024) and inp["logits"].dtype == np.float32
    assert inp["draft_tokens"].shape == (2, 3)
    assert list(inp["block_table"][0]) == [0, -1] and list(inp["block_table"][1]) == [1, 2]


def test_causal_bounds_formula():
    assert list(causal_bounds(np.array([10, 3]), 2)) == [8, 9, 10, 1, 2, 3]
    assert list(causal_bounds(np.array([5]), 0)) == [5]


@pytest.mark.parametrize("name", ["c2", "c3"])
def test_shuffled_tables_are_a_permutation(name):
    cfg = small_config(name, R=6, vocab=64)
    inp = make_inputs(cfg, seed=0)
    bt = inp["block_table"]
    ids = bt[bt >= 0]
    assert np.array_equal(np.sort(ids), np.arange(inp["num_pages"]))
    pages = -(-inp["kv_lens_in"] // 64)
    assert np.array_equal((bt >= 0).sum(axis=1), pages)
    assert np.all((inp["kv_lens_in"] >= 1024) & (inp["kv_lens_in"] <= 1536))


def test_c4_structure_small_vocab():
    cfg = small_config("c4", vocab=256)
    inp = make_inputs(cfg, seed=0)
    L = inp["kv_lens_in"]
    k = cfg.k
    assert np.all((L >= 8192) & (L <= 32768))
    straddle = ((L % 64) >= 1) & ((L % 64) <= k)
    assert straddle.sum() >= cfg.R // 2
    assert len(inp["zero_bound_tokens"]) == round(0.1 * cfg.T)
    assert np.all(inp["kv_bounds"][inp["zero_bound_tokens"]] == 0)
    nz = np.setdiff1d(np.arange(cfg.T), inp["zero_bound_tokens"])
    expect = causal_bounds(L, k)
    assert np.array_equal(inp["kv_bounds"][nz], expect[nz])


def test_planted_maximum_and_draft_rate():
    cfg = small_config("c1", R=64, vocab=4096, kv_lens=None, kv_len_range=(64, 128))
    inp = make_inputs(cfg, seed=0)
    x = inp["logits"]
    T = cfg.T
    planted = inp["planted_argmax"]
    assert np.all(x[np.arange(T), planted] == np.float32(12.0))
    others = x.copy()
    others[np.arange(T), planted] = -np.inf
    assert np.all(others.max(axis=1) <= 11.0)
    k = cfg.k
    match = np.array([[inp["draft_tokens"][r, j] == planted[r * (k + 1) + j] for j in range(k)]
                      for r in range(cfg.R)])
    assert 0.5 < match.mean() < 0.7


def test_config_table():
    assert CONFIGS["c1"].T == 8 and CONFIGS["c2"].T == 160 and CONFIGS["c3"].T == 64
    assert CONFIGS["c4"].T == 128 and CONFIGS["c0"].T == 8
    for c in CONFIGS.values():
        assert c.D == 512 and c.page_size == 64
        assert abs(c.softmax_scale - 128 ** -0.5) < 1e-15
