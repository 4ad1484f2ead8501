"""The float64 oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle)


@pytest.mark.parametrize("pin", pins.SAMPLED_PINS, ids=lambda f: f.__name__)
def test_sampled_pin(pin):
    pin(oracle)


def test_bf16_rounding():
    pins.check_bf16_rounding()


def test_combine_all_empty_rows_no_nan():
    po = np.zeros((3, 2, 1, 4))
    pl = np.full((3, 2, 1), -np.inf)
    pl[1, 1, 0] = 0.25
    po[1, 1, 0] = [1, 2, 3, 4]
    o, l = oracle.ref_lse_combine(po, pl)
    assert l[0, 0] == -np.inf and np.all(o[0, 0] == 0)
    assert l[1, 0] == 0.25 and np.allclose(o[1, 0], [1, 2, 3, 4])


def test_greedy_rejects_nonfinite():
    logits = np.zeros((2, 4), dtype=np.float32)
    logits[1, 2] = np.nan
    with pytest.raises(ValueError):
        oracle.ref_greedy_verify(logits, np.zeros((1, 1), np.int32), np.array([4]), 1)


def test_regression_fixture_c0():
    """The oracle still reproduces its recorded c0 results (tests/golden)."""
    import os
    from workloads import make_inputs
    path = os.path.join(os.path.dirname(__file__), "golden", "c0_oracle.txt")
    rows = {}
    for line in open(path):
        if line.startswith("#"):
            continue
        parts = line.split()
        rows.setdefault(parts[0], []).append(parts[1:])
    ref = oracle.ref_verify_step(make_inputs("c0", seed=0))
    for t, vals in enumerate(rows["lse"]):
        assert int(vals[0]) == t
        assert np.allclose(ref["lse"][t], [float(v) for v in vals[1:]], rtol=1e-13, atol=0)
    for t, vals in enumerate(rows["outsum"]):
        assert np.allclose(ref["out"][t].sum(axis=1), [float(v) for v in vals[1:]], rtol=1e-12, atol=1e-13)
    for key in ("argmax", "accepted", "next_tokens", "kv_lens_out"):
        assert [int(v) for v in rows[key][0]] == [int(v) for v in ref[key]], key
