"""The C ABI library: it builds, loads and exports every declared symbol, and
its host-side argument checks reject bad calls before any launch (CPU only:
no call here reaches the GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verify_mla_gb300 import build as B
    B.build()
    from speculative_decoding_verify_mla_gb300 import load_library
    return load_library()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([A-Za-z_]\w*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for f in ("mla_verify_decode", "mla_lse_combine", "spec_verify_greedy"):
        assert f in names


def test_every_declared_symbol_is_exported(lib):
    from speculative_decoding_verify_mla_gb300 import EXPORTED_SYMBOLS
    names = declared_functions()
    assert set(EXPORTED_SYMBOLS) <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    from speculative_decoding_verify_mla_gb300 import status_string
    assert status_string(0) == "ok"
    assert "workspace" in status_string(4)
    assert status_string(99) == "unknown status"


def test_workspace_queries(lib):
    from speculative_decoding_verify_mla_gb300 import attention_workspace_bytes, greedy_workspace_bytes
    assert attention_workspace_bytes(8, 64, 1) == 0
    assert attention_workspace_bytes(8, 64, 3) == 3 * 8 * 64 * (512 * 2 + 4)  # bf16 part_o + fp32 part_lse
    assert greedy_workspace_bytes(8, 163840) >= 256 + 8 * 8
    assert greedy_workspace_bytes(0, 10) == 256


def _attn_call(lib, **kw):
    args = dict(q=1 << 12, kv=1 << 12, num_pages=4, page_size=64, bt=1 << 12, R=2, qpr=4, maxp=2,
                bounds=1 << 12, gate=1 << 12, H=8, scale=0.1, splits=1, ws=None, ws_bytes=0,
                out=1 << 12, lse=1 << 12, status=None, stream=None)
    args.update(kw)
    return lib.mla_verify_decode(args["q"], args["kv"], args["num_pages"], args["page_size"], args["bt"],
                                 args["R"], args["qpr"], args["maxp"], args["bounds"], args["gate"],
                                 args["H"], ctypes.c_float(args["scale"]), args["splits"], args["ws"],
                                 args["ws_bytes"], args["out"], args["lse"], args["status"], args["stream"])


def test_attention_host_checks(lib):
    # every failure below is decided before any CUDA call
    assert _attn_call(lib, page_size=32) == 5          # unsupported page size
    assert _attn_call(lib, R=-1) == 2
    assert _attn_call(lib, qpr=0) == 2
    assert _attn_call(lib, H=0) == 2
    assert _attn_call(lib, splits=65) == 2
    assert _attn_call(lib, R=0) == 0                  # empty batch: nothing to do
    assert _attn_call(lib, scale=float("nan")) == 2
    assert _attn_call(lib, scale=-1.0) == 2
    assert _attn_call(lib, num_pages=0) == 2
    assert _attn_call(lib, q=None) == 1
    assert _attn_call(lib, lse=None) == 1
    assert _attn_call(lib, q=(1 << 12) + 8) == 3       # q must be 16-byte aligned
    assert _attn_call(lib, out=(1 << 12) + 2) == 3


def test_combine_host_checks(lib):
    assert lib.mla_lse_combine(None, None, 0, 1, 1, None, None, None, None) == 2
    assert lib.mla_lse_combine(None, None, 2, 0, 8, None, None, None, None) == 0
    assert lib.mla_lse_combine(None, 4096, 2, 1, 8, 4096, 4096, 4096, None) == 1
    assert lib.mla_lse_combine(4096 + 4, 4096, 2, 1, 8, 4096, 4096, 4096, None) == 3


def test_greedy_host_checks(lib):
    f = lib.spec_verify_greedy
    assert f(4096, 7, 10, 2, 3, 4096, 4096, 4096, 4096, 4096, 4096, 4096, 1 << 20, None) == 2  # T != R(k+1)
    assert f(4096, 0, 10, 0, 3, None, None, None, None, None, None, None, 0, None) == 0
    assert f(4096, 8, 0, 2, 3, 4096, 4096, 4096, 4096, 4096, 4096, 4096, 1 << 20, None) == 2  # V = 0
    assert f(None, 8, 10, 2, 3, 4096, 4096, 4096, 4096, 4096, 4096, 4096, 1 << 20, None) == 1
    assert f(4096, 8, 10, 2, 3, None, 4096, 4096, 4096, 4096, 4096, 4096, 1 << 20, None) == 1  # drafts
    assert f(4096, 8, 10, 2, 3, 4096, 4096, 4096, 4096, 4096, 4096, 4096, 8, None) == 4      # workspace
    assert f(4096, 8, 10, 2, 3, 4096, 4096, 4096, 4096, 4096, 4096, 4096 + 16, 1 << 20, None) == 3


def test_kv_append_host_checks(lib):
    f = lib.mla_kv_append
    assert f(4096, 4096, 4096, 2, 4, 2, 4096, 4, 32, None, None) == 5   # page size
    assert f(4096, 4096, 4096, -1, 4, 2, 4096, 4, 64, None, None) == 2
    assert f(4096, 4096, 4096, 0, 4, 2, 4096, 4, 64, None, None) == 0   # nothing to do
    assert f(None, 4096, 4096, 2, 4, 2, 4096, 4, 64, None, None) == 1
    assert f(4096 + 8, 4096, 4096, 2, 4, 2, 4096, 4, 64, None, None) == 3


def test_sampled_host_checks(lib):
    f = lib.spec_verify_sampled
    fl = ctypes.c_float
    ws = lib.sv_sampled_workspace_bytes(2, 3, 1000)
    assert ws >= 256
    args = [4096, 2, 3, 1000, fl(1.0), 4096, 4096, 4096, 4096, 4096, 4096, 4096, 4096, ws, None]
    bad = list(args); bad[4] = fl(0.0)
    assert f(*bad) == 2                     # temperature must be > 0
    bad = list(args); bad[4] = fl(float("inf"))
    assert f(*bad) == 2
    bad = list(args); bad[3] = 0
    assert f(*bad) == 2                     # V >= 1
    bad = list(args); bad[1] = 0
    assert f(*bad) == 0                     # no requests: nothing to do
    bad = list(args); bad[6] = None
    assert f(*bad) == 1                     # draft_probs needed when k > 0
    bad = list(args); bad[13] = ws - 1
    assert f(*bad) == 4
    bad = list(args); bad[12] = 4096 + 16
    assert f(*bad) == 3                     # workspace 256-byte aligned


def test_balanced_plan_host_checks(lib):
    assert _attn_call(lib, splits=-3) == 2                       # only -1 and -2 are valid negatives
    assert _attn_call(lib, splits=-1) == 4                       # the plan needs a workspace
    assert _attn_call(lib, splits=-1, maxp=70000) == 2           # piece bounds are 16-bit
    from speculative_decoding_verify_mla_gb300 import SV_SPLITS_BALANCED, attention_workspace_bytes
    assert SV_SPLITS_BALANCED == -1
    assert attention_workspace_bytes(128, 64, -1) > 128 * 64 * 2052


def test_auto_split_choice(lib):
    from speculative_decoding_verify_mla_gb300 import SV_SPLITS_WAVE, attention_workspace_bytes, num_splits_for
    assert num_splits_for(1, 8, 64, 24) >= 1       # one request: uniform splits
    assert num_splits_for(16, 8, 64, 512) == -1    # long contexts, one wave: balanced plan
    # 32 requests x 3 row tiles x 2 halves = 192 CTAs: between one and two
    # waves of the (fallback) 152 SMs -> the wave mode
    assert num_splits_for(32, 5, 64, 24) == SV_SPLITS_WAVE == -2
    assert num_splits_for(64, 1, 64, 24) >= 1      # 128 CTAs (stacked form): uniform splits
    assert num_splits_for(20, 5, 64, 24) >= 1      # 120 CTAs fit one wave: uniform splits
    assert num_splits_for(60, 5, 64, 24) >= 1      # 360 CTAs: more than two waves
    assert attention_workspace_bytes(160, 64, -2) >= 7 * 3 * 320 * (1024 + 4)  # the split requests' slots


def test_form_is_per_call(lib):
    """The kernel form is an argument of each call (no process-wide state):
    the split query takes it, unknown forms are rejected, and the stacked
    form changes the automatic split count for requests of <= 64 query rows
    (one CTA per unit instead of two, when the units stay >= 4 tiles long);
    larger requests are unaffected."""
    import speculative_decoding_verify_mla_gb300 as sv
    sms = 152  # no device here: the library's fallback SM count
    auto = sv.num_splits_for(64, 1, 64, 24, sv.FORM_AUTO)
    short = sv.num_splits_for(2, 4, 8, 2, sv.FORM_AUTO)
    always_short = sv.num_splits_for(2, 4, 8, 8, sv.FORM_STACKED)
    off = sv.num_splits_for(64, 1, 64, 24, sv.FORM_TWO_CTA)
    off_short = sv.num_splits_for(2, 4, 8, 8, sv.FORM_TWO_CTA)
    wide_auto = sv.num_splits_for(1, 8, 64, 24, sv.FORM_AUTO)
    wide_off = sv.num_splits_for(1, 8, 64, 24, sv.FORM_TWO_CTA)
    assert auto == min(sms // 64, 24 // 2) and off == min(sms // 128, 24 // 2)
    assert short == 1                              # 2-page units: the two-CTA form, 1 split
    assert always_short == 4 and off_short == 4    # 8 pages: min(SMs / CTAs per split, 8 / 2)
    assert wide_auto == wide_off
    # the calls' answers do not depend on the order they were made in
    assert sv.num_splits_for(64, 1, 64, 24, sv.FORM_AUTO) == auto
    with pytest.raises(ValueError):
        sv.num_splits_for(64, 1, 64, 24, 7)
    assert lib.sv_mla_verify_num_splits(64, 1, 64, 24, -1) == 0


def test_gated_and_wuv_host_checks(lib):
    args = dict(q=1 << 12, kv=1 << 12, num_pages=4, page_size=64, bt=1 << 12, R=2, qpr=4, maxp=2,
                bounds=1 << 12, gate=1 << 12, H=8, scale=0.1, splits=1, ws=None, ws_bytes=0,
                out=1 << 12, lse=1 << 12, status=None, stream=None)

    def gated(gate_dim, **kw):
        a = dict(args)
        a.update(kw)
        return lib.mla_verify_decode_gated(a["q"], a["kv"], a["num_pages"], a["page_size"], a["bt"], a["R"],
                                           a["qpr"], a["maxp"], a["bounds"], a["gate"], gate_dim, a["H"],
                                           ctypes.c_float(a["scale"]), a["splits"], a.get("form", 0), a["ws"],
                                           a["ws_bytes"], a["out"], a["lse"], a["status"], a["stream"])
    assert gated(7) == 5          # gate_dim must be 512 or 1
    assert gated(1, form=3) == 5  # unknown kernel form
    assert gated(1, form=-1) == 5
    assert gated(1, R=0) == 0
    assert gated(1, q=None) == 1
    f = lib.mla_wuv_project
    assert f(4096, 4096, 4, 2, 100, 4096, None, None) == 5   # v_dim not a multiple of 32
    assert f(4096, 4096, 4, 2, 512, 4096, None, None) == 5   # v_dim > 256
    assert f(4096, 4096, 0, 2, 128, 4096, None, None) == 0
    assert f(None, 4096, 4, 2, 128, 4096, None, None) == 1
    assert f(4096 + 8, 4096, 4, 2, 128, 4096, None, None) == 3


def test_kv8_host_checks(lib):
    f = lib.mla_verify_decode_kv8
    fl = ctypes.c_float
    base = [1 << 12, 1 << 12, fl(0.5), 4, 64, 1 << 12, 2, 4, 2, 1 << 12, 1 << 12, 512, 8, fl(0.1), 1, 0,
            None, 0, 1 << 12, 1 << 12, None, None]
    a = list(base); a[2] = fl(0.0)
    assert f(*a) == 2            # kv_scale must be > 0
    a = list(base); a[2] = fl(float("nan"))
    assert f(*a) == 2
    a = list(base); a[4] = 32
    assert f(*a) == 5            # page size
    a = list(base); a[1] = None
    assert f(*a) == 1
    a = list(base); a[6] = 0
    assert f(*a) == 0            # no requests
    a = list(base); a[15] = 9
    assert f(*a) == 5            # unknown kernel form


def test_wait_limit_entry_only_shortens_the_waits(lib):
    """The test entry point with a per-call wait limit refuses a limit above
    the library's own two seconds before it looks at any other argument
    (every pointer here is NULL)."""
    f = lib.sv_test_mla_verify_decode_wait_limit
    c = ctypes
    f.argtypes = [c.c_void_p, c.c_void_p, c.c_int, c.c_float, c.c_int, c.c_int, c.c_void_p, c.c_int, c.c_int,
                  c.c_int, c.c_void_p, c.c_void_p, c.c_int, c.c_int, c.c_float, c.c_int, c.c_int, c.c_void_p,
                  c.c_size_t, c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p, c.c_uint64]
    f.restype = c.c_int
    args = [None, None, 0, 1.0, 4, 64, None, 2, 4, 2, None, None, 512, 8, 0.1, 1, 0, None, 0, None, None, None,
            None]
    assert f(*args, 2_000_000_001) == 2  # SV_ERR_SHAPE
    assert f(*args, (1 << 64) - 1) == 2
    for limit in (0, 1000, 2_000_000_000):
        assert f(*args, limit) == 1  # SV_ERR_NULL: the usual checks follow
    g = lib.sv_test_mla_wuv_project_wait_limit
    g.argtypes = [c.c_void_p, c.c_void_p, c.c_int, c.c_int, c.c_int, c.c_void_p, c.c_void_p, c.c_void_p,
                  c.c_uint64]
    g.restype = c.c_int
    assert g(None, None, 8, 4, 128, None, None, None, 2_000_000_001) == 2  # SV_ERR_SHAPE
    for limit in (0, 2_000_000_000):
        assert g(None, None, 8, 4, 128, None, None, None, limit) == 1  # SV_ERR_NULL
