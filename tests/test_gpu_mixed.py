"""GPU parity of the mixed NVFP4/FP8 route against the oracle (FLAMIA technical
review section 2, "the mixed route"; Korean review section 3.1; readings C-7,
C-8).

NVFP4 score operands (E2M1 codes, E4M3 group scales), the per-token V copy of
the diagonal key tiles and the E4M3 token-block copies: bit-exact; O, dQ, dK
and dV within 1e-2 normalised max-abs error, LSE within 1e-3; and the route's
locality: a
change to any later token leaves every earlier row's O and LSE bit-identical.
"""
import numpy as np
import pytest

import flamia_workloads as W
import oracle as O
from gpu_harness import run_gpu, run_oracle
from metrics import cosine, norm_max_err

pytestmark = pytest.mark.gpu
TOL = 1e-2
MIXED = O.Options(mixed=True)


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from microscaled_precision_causal_gb300 import build
    build.build()


def _unpack(packed):
    return np.stack([packed & 0x0F, packed >> 4], axis=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)


CASES = [
    ("ragged_gqa_outliers", [300, 77, 129, 1], 2, 1, 0, "normal_outliers"),
    ("two_docs_gqa4", [200, 517], 4, 1, 0, "normal"),
    ("mha_tail", [130, 5, 260], 2, 2, 19, "student_t3"),
]


@pytest.mark.parametrize("name,lengths,hq,hkv,extra,dist", CASES, ids=[c[0] for c in CASES])
def test_mixed_training_call_matches_oracle(name, lengths, hq, hkv, extra, dist):
    d = 128
    T = sum(lengths) + extra
    w = W.custom([T], hq, hkv, d, dist=dist, seed=51)
    inp = W.make_inputs(w)
    g = run_gpu(inp, lengths, hq, hkv, d, total_tokens=T, mixed=True)
    o = run_oracle(inp, lengths, hq, hkv, d, opts=MIXED)
    assert g["status"] == 0
    valid = sum(lengths)
    for n in ("q", "k"):
        assert np.array_equal(_unpack(g[n + "4_codes"])[:valid], o[n + "_nvfp4_codes"][:valid]), n
        assert np.array_equal(g[n + "4_scales"][:valid], o[n + "_nvfp4_scales"][:valid]), n
    assert np.array_equal(g["vt_codes"], o["v_tok_codes"]) and np.array_equal(g["vt_scales"], o["v_tok_scales"])
    for n in ("q", "k", "v"):
        assert np.array_equal(g[n + "_codes"], o[n + "_codes"]), n
    assert np.max(np.abs(g["lse"][:, :valid] - o["lse"][:, :valid])) < 1e-3
    assert np.array_equal(g["do_codes"], o["do_codes"]) and np.array_equal(g["do_scales"], o["do_scales"])
    msgs, worst = [], 0.0
    for n in ("o", "dq", "dk", "dv"):
        e = norm_max_err(g[n][:valid], o[n][:valid])
        worst = max(worst, e)
        msgs.append(f"{n}: err {e:.2e} cos {cosine(g[n][:valid], o[n][:valid]):.6f}")
    assert worst <= TOL, "; ".join(msgs)
    assert np.all(g["o"][valid:] == 0) and np.all(np.isinf(g["lse"][:, valid:]))
    for n in ("dq", "dk", "dv"):
        assert np.all(g[n][valid:] == 0), n


def test_mixed_forward_earlier_rows_are_bit_identical():
    """Any later token of Q, K or V (x 2^12) leaves O and LSE of every earlier
    row bit-identical: NVFP4 scales stay inside one token and the diagonal key
    tile takes V per key."""
    lengths, hq, hkv, d = [290, 60], 2, 1, 128
    w = W.custom(lengths, hq, hkv, d, seed=52)
    inp = W.make_inputs(w)
    base = run_gpu(inp, lengths, hq, hkv, d, with_bwd=False, mixed=True)
    for t in (1, 40, 150, 289):
        for name in ("q", "k", "v"):
            pert = {k_: v_.copy() for k_, v_ in inp.items()}
            pert[name][t] = W.f32_to_bf16_bits(W.bf16_bits_to_f32(pert[name][t]) * 2.0 ** 12)
            c = run_gpu(pert, lengths, hq, hkv, d, with_bwd=False, mixed=True)
            assert np.array_equal(c["o"][:t], base["o"][:t]), (name, t)
            assert np.array_equal(c["lse"][:, :t], base["lse"][:, :t]), (name, t)
            assert not np.array_equal(c["o"][t:290], base["o"][t:290]), (name, t)


def test_mixed_full_size_sampled():
    """B=4 x 8192, 32 query heads on 8 K/V heads, N(0,1) with 0.1% x100
    outliers, in the benchmark's launch configuration; the oracle recomputes
    the last document's last head group on sampled tiles (the backward of a
    sampled tile needs the forward LSE of every query tile it meets)."""
    wl = W.WORKLOADS["mixed_nvfp4_gqa_b4_s8192"]
    inp = W.make_inputs(wl)
    g = run_gpu(inp, list(wl.lengths), wl.hq, wl.hkv, wl.d, mixed=True)
    assert g["status"] == 0
    lengths = list(wl.lengths)
    n = len(lengths) - 1
    s0 = int(np.sum(lengths[:n])); L = lengths[n]; s1 = s0 + L
    hk = wl.hkv - 1
    gsz = wl.hq // wl.hkv
    heads = list(range(hk * gsz, (hk + 1) * gsz))
    sub = {name: arr[s0:s1][:, heads if name in ("q", "do") else [hk]] for name, arr in inp.items()}
    nt = -(-L // 128)
    sel = dict(q_tiles={0: [0, 1, nt - 2, nt - 1]}, k_tiles={0: [nt - 2, nt - 1]}, bwd_q_tiles={0: [1, nt - 1]})
    o = run_oracle(sub, [L], gsz, 1, wl.d, opts=MIXED, **sel)
    rows_o = np.r_[0:256, (nt - 2) * 128:L]
    rows_q = np.r_[128:256, (nt - 1) * 128:L]
    rows_k = np.r_[(nt - 2) * 128:L]
    gl = {key: (g[key][s0:s1][:, heads] if key in ("o", "dq") else g[key][s0:s1][:, [hk]]) for key in
          ("o", "dq", "dk", "dv")}
    for key, rows in (("o", rows_o), ("dq", rows_q), ("dk", rows_k), ("dv", rows_k)):
        e = norm_max_err(gl[key][rows], o[key][rows])
        assert e <= TOL, f"{key}: {e:.3e} cos {cosine(gl[key][rows], o[key][rows]):.6f}"
    assert np.max(np.abs(g["lse"][heads][:, s0:s1][:, rows_o] - o["lse"][:, rows_o])) < 1e-3
