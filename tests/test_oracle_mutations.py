"""Plant a mistake in (a copy of) the oracle and check that some pin fails.

This shows the pins are strong enough to catch the plausible slips: an
off-by-one bound, a dropped softmax scale, a flipped gate sign, a wrong
token -> request mapping, a base-2 LSE, the last index on argmax ties, a draft
compared with the wrong target position, a wrong trim, an unnormalised merge
weight and a NaN instead of the (-inf, 0) identity.  Mutations live on the CPU
and only ever in a private copy of the oracle module.
"""
import importlib.util
import sys

import numpy as np
import pytest

import pins


def _fresh_oracle():
    spec = importlib.util.find_spec("oracle.verify_ref")
    mod = importlib.util.module_from_spec(spec)
    sys.modules["_oracle_mutant"] = mod
    spec.loader.exec_module(mod)
    return mod


def _mut_bound_off_by_one(m):
    orig = m.ref_verify_attention

    def f(q, kv, bt, b, g, qpr, scale):
        # each token also sees the position right after its own
        b = np.asarray(b).copy()
        for t in range(b.shape[0]):
            cap = int(np.sum(np.asarray(bt[t // qpr]) >= 0)) * kv.shape[1]
            if b[t] > 0:
                b[t] = min(b[t] + 1, cap)
        return orig(q, kv, bt, b, g, qpr, scale)
    m.ref_verify_attention = f


def _mut_no_scale(m):
    orig = m.ref_verify_attention
    m.ref_verify_attention = lambda q, kv, bt, b, g, qpr, scale: orig(q, kv, bt, b, g, qpr, 1.0)


def _mut_gate_sign(m):
    orig = m.sigmoid
    m.sigmoid = lambda x: orig(-np.asarray(x, dtype=np.float64))


def _mut_token_mapping(m):
    orig = m.ref_verify_attention

    def f(q, kv, bt, b, g, qpr, scale):
        # tokens interleaved across requests instead of request-major
        T = np.asarray(b).shape[0]
        R = max(1, T // qpr)
        order = np.array([(t % R) * qpr + t // R for t in range(T)])
        out, lse = orig(np.asarray(q)[order], kv, bt, np.asarray(b)[order], np.asarray(g)[order], qpr, scale)
        inv = np.argsort(order)
        return out[inv], lse[inv]
    m.ref_verify_attention = f


def _mut_lse_log2(m):
    orig = m._softmax_stats

    def f(s, rows):
        lse, o = orig(s, rows)
        return lse / np.log(2.0), o
    m._softmax_stats = f


def _mut_argmax_last(m):
    def f(logits, drafts, kv_in, k):
        x = np.asarray(logits, dtype=np.float64)
        a = x.shape[1] - 1 - np.argmax(x[:, ::-1], axis=1)
        R = len(kv_in)
        n = np.zeros(R, np.int64)
        for r in range(R):
            while n[r] < k and drafts[r][n[r]] == a[r * (k + 1) + n[r]]:
                n[r] += 1
        return a, n, a[np.arange(R) * (k + 1) + n], np.asarray(kv_in) - (k - n)
    m.ref_greedy_verify = f


def _mut_draft_position(m):
    def f(logits, drafts, kv_in, k):
        a = np.argmax(np.asarray(logits, dtype=np.float64), axis=1)
        R = len(kv_in)
        n = np.zeros(R, np.int64)
        for r in range(R):
            while n[r] < k and drafts[r][n[r]] == a[r * (k + 1) + n[r] + 1]:
                n[r] += 1
        return a, n, a[np.arange(R) * (k + 1) + n], np.asarray(kv_in) - (k - n)
    m.ref_greedy_verify = f


def _mut_trim(m):
    orig = m.ref_greedy_verify

    def f(logits, drafts, kv_in, k):
        a, n, nxt, kv = orig(logits, drafts, kv_in, k)
        return a, n, nxt, np.asarray(kv_in) - n
    m.ref_greedy_verify = f


def _mut_unnormalised_merge(m):
    def f(part_o, part_lse, gate=None):
        part_o = np.asarray(part_o, dtype=np.float64)
        part_lse = np.asarray(part_lse, dtype=np.float64)
        m_ = part_lse.max(axis=0)
        empty = ~np.isfinite(m_)
        ms = np.where(empty, 0.0, m_)
        w = np.where(empty[None], 0.0, np.exp(part_lse - ms[None]))
        z = w.sum(axis=0)
        lse = np.where(empty, -np.inf, ms + np.log(np.where(empty, 1.0, z)))
        o = (w[..., None] * part_o).sum(axis=0)
        if gate is not None:
            o = m.sigmoid(m._as_f64(gate)) * o
        return o, lse
    m.ref_lse_combine = f


def _mut_nan_identity(m):
    orig = m._softmax_stats

    def f(s, rows):
        if s.shape[1] == 0:
            return np.full(s.shape[0], -np.inf), np.full((s.shape[0], rows.shape[1]), np.nan)
        return orig(s, rows)
    m._softmax_stats = f


def _mut_wuv_wrong_head(m):
    orig = m.ref_wuv_project
    m.ref_wuv_project = lambda x, w: orig(x, np.roll(m._as_f64(w), 1, axis=0))


def _mut_headwise_gate_ignored(m):
    orig = m.gate_factor
    m.gate_factor = lambda g: np.ones((len(g), 1)) if np.asarray(g).ndim == 1 else orig(g)


def _mut_wuv_transposed_input(m):
    def f(x, w):
        x = m._as_f64(x)
        w = m._as_f64(w)
        v = np.zeros((x.shape[0], x.shape[1], w.shape[1]))
        for h in range(x.shape[1]):
            v[:, h, :] = x[:, h, ::-1] @ w[h].T  # latent columns reversed
        return v
    m.ref_wuv_project = f


def _mut_e4m3_bias(m):
    orig = m.e4m3_bits_to_f64
    m.e4m3_bits_to_f64 = lambda c: orig(c) * 0.5  # exponent bias 8 instead of 7


MUTATIONS = [
    _mut_e4m3_bias,
    _mut_wuv_wrong_head, _mut_headwise_gate_ignored, _mut_wuv_transposed_input,
    _mut_bound_off_by_one, _mut_no_scale, _mut_gate_sign, _mut_token_mapping, _mut_lse_log2,
    _mut_argmax_last, _mut_draft_position, _mut_trim, _mut_unnormalised_merge, _mut_nan_identity,
]


@pytest.mark.parametrize("mutate", MUTATIONS, ids=lambda f: f.__name__)
def test_some_pin_catches(mutate):
    m = _fresh_oracle()
    mutate(m)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(m)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught {mutate.__name__}"


# --------------------------------------------------------------------------
# sampled verification: each mutation rewrites one expression of a private
# copy of the sampled-verification oracle's source
# --------------------------------------------------------------------------
SAMPLED_MUTATIONS = {
    "residual_not_clipped": ("w = np.maximum(p - qd[r, j], 0.0)", "w = p - qd[r, j]"),
    "residual_is_target": ("w = np.maximum(p - qd[r, j], 0.0)", "w = p.copy()"),
    "ratio_inverted": ("lhs, rhs = u[r, j] * qd[r, j, d], p[d]", "lhs, rhs = u[r, j] * p[d], qd[r, j, d]"),
    "bonus_wrong_row": ("w = target_probs(x[base + k], temperature)",
                        "w = target_probs(x[base + k - 1], temperature)"),
    "cdf_left_side": ('side="right"', 'side="left"'),
    "temperature_multiplies": ("/ float(temperature)", "* float(temperature)"),
    "trim_wrong": ("int(kv_lens_in[r]) - (k - n)", "int(kv_lens_in[r]) - n"),
    "accepted_counts_rejected": ("            n = j\n", "            n = j + 1\n"),
}


def _sampled_mutant(old, new):
    import types
    spec = importlib.util.find_spec("oracle.sampled_ref")
    src = open(spec.origin).read()
    assert src.count(old) >= 1, old
    mod = types.ModuleType("_sampled_mutant")
    exec(compile(src.replace(old, new), spec.origin, "exec"), mod.__dict__)
    # the greedy oracle is needed by the greedy-limit pin
    import oracle
    mod.ref_greedy_verify = oracle.ref_greedy_verify
    return mod


@pytest.mark.parametrize("name", sorted(SAMPLED_MUTATIONS))
def test_some_sampled_pin_catches(name):
    m = _sampled_mutant(*SAMPLED_MUTATIONS[name])
    caught = []
    for pin in pins.SAMPLED_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(m)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught {name}"
