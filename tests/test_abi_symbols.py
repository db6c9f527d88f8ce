"""The C-ABI library builds for sm_103a, loads, and exports every function that
include/flamia.h declares.  Host-side argument validation is exercised on the
paths that return before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "flamia.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(flamia_[a-z0-9_]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def flamia():
    from microscaled_precision_causal_gb300 import build
    build.build()
    import microscaled_precision_causal_gb300 as F
    return F


def test_header_declares_the_three_named_entry_points():
    names = _declared_functions()
    for n in ("flamia_quantize_tokenblock", "flamia_fwd", "flamia_bwd"):
        assert n in names


def test_library_exports_every_declared_symbol(flamia):
    L = flamia.lib()
    for name in _declared_functions():
        assert hasattr(L, name), name
    assert set(flamia.EXPORTED) == set(_declared_functions())


def test_host_validation_without_gpu(flamia):
    L = flamia.lib()
    F = flamia
    assert L.flamia_status_string(0) == b"ok"
    assert L.flamia_plan_bytes(-1, 1) == 0
    assert L.flamia_plan_bytes(1024, 3) > 1024 // 128 * 32
    assert L.flamia_bwd_workspace_bytes(1000, 2, 4, 2, 128) >= 1000 * 4 * 128 * 3
    q = F.QTensor(16, 16, None)
    o = F.default_options()
    assert (o.p_boost_log2, o.bwd_p_boost_log2, o.dq_headroom_log2) == (8, 8, 14)
    args = lambda **kw: dict(dict(hq=4, hkv=2, d=128, causal=1, opts=o, plan=256, out=256, lse=256), **kw)

    def fwd(a):
        return L.flamia_fwd(ctypes.byref(q), ctypes.byref(q), ctypes.byref(q), 256, 1, 100, a["hq"], a["hkv"], a["d"],
                            a["causal"], 0.0, ctypes.byref(a["opts"]), a["plan"], a["out"], a["lse"], None)
    assert fwd(args(d=96)) == -2                      # unsupported head dim
    assert fwd(args(hq=3)) == -2                      # hq % hkv != 0
    assert fwd(args(causal=2)) == -1                  # causal is 0 or 1
    strict_nc = F.default_options()
    for f in ("strict_per_token", "strict_row_ds", "strict_causal_dq"):
        setattr(strict_nc, f, 1)
    assert fwd(args(causal=0, opts=strict_nc)) == -2  # the strict options are causal only
    sw = F.default_options(); sw.window_left = 64
    for f in ("strict_per_token", "strict_row_ds", "strict_causal_dq"):
        setattr(sw, f, 1)
    assert fwd(args(opts=sw)) == -2                   # ... and take no sliding window
    assert (o.window_left, o.window_right) == (-1, -1)
    assert fwd(args(plan=0)) == -1                    # null plan
    assert fwd(args(out=258)) == -3                   # misaligned output
    bad = F.default_options(); bad.p_boost_log2 = 10
    assert fwd(args(opts=bad)) == -2
    qm = F.QTensor(17, 16, None)                      # misaligned codes
    assert L.flamia_fwd(ctypes.byref(qm), ctypes.byref(q), ctypes.byref(q), 256, 1, 100, 4, 2, 128, 1, 0.0, None, 256,
                        256, 256, None) == -3
    assert L.flamia_quantize_tokenblock(256, 100, 2, 80, 256, 1, 256, 0, 256, 256, None, None) == -2
    assert L.flamia_plan_build(256, 1, 100, 256, 8, None) == -4     # plan buffer too small
    # backward needs k/v stats
    assert L.flamia_bwd(ctypes.byref(q), ctypes.byref(q), ctypes.byref(q), 256, 256, 256, 256, 1, 100, 4, 2, 128, 1,
                        0.0, None, 256, 256, 256, 256, 256, 1 << 30, None) == -1


def test_strict_options_come_as_a_set(flamia):
    """The strict options are accepted together (per-token scales, per-row dS
    exponents, causal dQ boost; deterministic may be added); a partial set, a
    deterministic flag without them, the mixed route without its operands or
    together with the strict options is refused before any CUDA call."""
    L, F = flamia.lib(), flamia
    q = F.QTensor(16, 16, None)

    def fwd(o):
        return L.flamia_fwd(ctypes.byref(q), ctypes.byref(q), ctypes.byref(q), 256, 1, 100, 4, 2, 128, 1, 0.0,
                            ctypes.byref(o), 256, 258, 256, None)   # misaligned output: reached only if opts pass
    for flags, want in ((("strict_per_token",), -2), (("strict_per_token", "strict_row_ds"), -2),
                        (("strict_causal_dq",), -2), (("deterministic",), -2), (("mixed_nvfp4",), -1),
                        (("mixed_nvfp4", "strict_per_token", "strict_row_ds", "strict_causal_dq"), -2),
                        (("strict_per_token", "strict_row_ds", "strict_causal_dq"), -3),
                        (("strict_per_token", "strict_row_ds", "strict_causal_dq", "deterministic"), -3)):
        o = F.default_options()
        for f in flags:
            setattr(o, f, 1)
        assert fwd(o) == want, flags


def test_backward_diagnostic_output_limits(flamia):
    """The fp32 P / dS diagnostic output of flamia_bwd is refused outside its
    scope (strict options, more than 1024 tokens) before any CUDA call."""
    L, F = flamia.lib(), flamia
    q = F.QTensor(16, 16, 16)

    def bwd(o, T):
        return L.flamia_bwd(ctypes.byref(q), ctypes.byref(q), ctypes.byref(q), 256, 256, 256, 256, 1, T, 4, 2, 128, 1,
                            0.0, ctypes.byref(o), 256, 256, 256, 256, 256, 1 << 30, None)
    o = F.default_options()
    o.debug_p_ds = 256
    assert bwd(o, 2000) == -2
    for f in ("strict_per_token", "strict_row_ds", "strict_causal_dq"):
        setattr(o, f, 1)
    assert bwd(o, 100) == -2


def test_dynamic_schedule_option_values(flamia):
    """The forward's work acquisition is 0 (static, the default) or 1 (cluster
    launch control); anything else is refused before any CUDA call."""
    L, F = flamia.lib(), flamia
    q = F.QTensor(16, 16, None)

    def fwd(o):
        return L.flamia_fwd(ctypes.byref(q), ctypes.byref(q), ctypes.byref(q), 256, 1, 100, 4, 2, 128, 1, 0.0,
                            ctypes.byref(o), 256, 258, 256, None)   # misaligned output: reached only if opts pass
    o = F.default_options()
    assert o.dynamic_schedule == 0
    for val, want in ((0, -3), (1, -3), (2, -2), (-1, -2)):
        o.dynamic_schedule = val
        assert fwd(o) == want, val
