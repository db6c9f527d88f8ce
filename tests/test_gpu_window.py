"""GPU parity of noncausal and windowed calls against the oracle.

The pages time packed noncausal training calls beside the causal ones (FLAMIA
review section 8 and its Appendix H; the batched 2 x 8192 noncausal case of
Appendix J; Korean review section 4.8).  A call's visible keys are a (left,
right) window per document: query i sees key j iff i - left <= j <= i + right
(-1: no limit); noncausal = (-1, -1).  Tolerance as for the causal calls: O,
dQ, dK, dV within 1e-2 of the oracle in normalised max-abs error, LSE within
1e-3, codes bit-exact.
"""
import numpy as np
import pytest

import flamia_workloads as W
import oracle as O
from gpu_harness import run_gpu, run_oracle
from metrics import cosine, norm_max_err

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from microscaled_precision_causal_gb300 import build
    build.build()


CASES = [
    # (name, lengths, hq, hkv, d, extra tokens past the last document, window)
    ("noncausal_ragged_gqa_d128", [300, 77, 129, 1], 2, 1, 128, 5, (-1, -1)),
    ("noncausal_mha_d64", [256, 130, 33], 2, 2, 64, 0, (-1, -1)),
    ("sliding_causal_100_d128", [700, 129, 40], 4, 2, 128, 3, (100, 0)),
    ("sliding_causal_300_d64", [517, 260], 2, 1, 64, 0, (300, 0)),
    ("two_sided_40_25_d128", [600, 128, 70], 2, 2, 128, 0, (40, 25)),
    ("right_only_3_d64", [400, 90], 2, 2, 64, 7, (3, -1)),
    ("left_only_unbounded_right_10_d128", [333, 256], 2, 1, 128, 0, (-1, 10)),
    ("wide_window_gqa8_d64", [640, 129], 8, 1, 64, 0, (200, 130)),
]


@pytest.mark.parametrize("name,lengths,hq,hkv,d,extra,window", CASES, ids=[c[0] for c in CASES])
def test_windowed_training_call_matches_oracle(name, lengths, hq, hkv, d, extra, window):
    T = sum(lengths) + extra
    inp = W.make_inputs(W.custom([T], hq, hkv, d, seed=31))
    g = run_gpu(inp, lengths, hq, hkv, d, total_tokens=T, window=window)
    o = run_oracle(inp, lengths, hq, hkv, d, opts=O.Options(window=window))
    assert g["status"] == 0
    for n in ("q", "k", "v"):
        assert np.array_equal(g[n + "_codes"], o[n + "_codes"]), n
    assert np.array_equal(g["do_codes"], o["do_codes"])
    valid = sum(lengths)
    assert np.max(np.abs(g["lse"][:, :valid] - o["lse"][:, :valid])) < 1e-3
    assert np.all(np.isinf(g["lse"][:, valid:]))
    for n in ("o", "dq", "dk", "dv"):
        e = norm_max_err(g[n], o[n])
        assert e <= TOL, f"{n}: {e:.3e} cos {cosine(g[n], o[n]):.6f}"
        assert np.all(g[n][valid:] == 0), n


@pytest.mark.parametrize("window", [(-1, -1), (300, 0), (40, 25)])
def test_windowed_plan_matches_oracle_work_lists(window):
    """flamia_plan_build_window orders the items by the window's costs exactly as
    the oracle's Algorithm 2 does."""
    import torch
    import microscaled_precision_causal_gb300 as F
    from gpu_harness import cu_tensor
    lengths = [1000, 200, 1, 3799, 130, 0, 640]
    T, N = sum(lengths), len(lengths)
    cu = cu_tensor(lengths)
    plan = torch.zeros(F.flamia_plan_bytes(T, N), dtype=torch.uint8, device="cuda")
    F.flamia_plan_build_window(cu, N, T, int(window[1] == 0), window[0], window[1], plan)
    torch.cuda.synchronize()
    w = plan.view(torch.int32).cpu().numpy()
    assert w[0] == 0
    nf, nb = int(w[6]), int(w[7])
    pref = ((16 + 3 * (N + 1) + 3) // 4) * 4
    cap = T // 128 + N + 1
    items = w[pref:pref + 4 * cap].reshape(cap, 4)[:nf]
    bitems = w[pref + 4 * cap:pref + 8 * cap].reshape(cap, 4)[:nb]
    cuh = np.concatenate([[0], np.cumsum(lengths)])
    want = O.work_list(cuh, window=window)
    assert [tuple(x) for x in items] == [(i["doc"], i["tile0"], i["ntiles"], i["cost"]) for i in want]
    bwant = O.bwd_key_tile_list(cuh, window=window)
    assert [tuple(x[:3]) for x in bitems] == [(b["doc"], b["ktile"], b["cost"]) for b in bwant]


@pytest.mark.parametrize("wname", ["noncausal_packed_16k_h16_d128", "noncausal_b2_s8192_h16_d128"])
def test_noncausal_full_size_sampled_parity(wname):
    """The full noncausal workload in the benchmark's launch configuration; the
    oracle recomputes the longest document x the last kv-head group: its whole
    forward, and the gradients of sampled tiles (every key tile of a sampled
    query tile, every query tile of a sampled key tile)."""
    w = W.WORKLOADS[wname]
    inp = W.make_inputs(w)
    lengths = list(w.lengths)
    g = run_gpu(inp, lengths, w.hq, w.hkv, w.d, window=w.window)
    assert g["status"] == 0
    n = int(np.argmax(lengths))
    s0 = int(np.sum(lengths[:n])); L = lengths[n]; s1 = s0 + L
    hk = w.hkv - 1
    gsz = w.hq // w.hkv
    heads = list(range(hk * gsz, (hk + 1) * gsz))
    sub = {name: arr[s0:s1][:, heads if name in ("q", "do") else [hk]] for name, arr in inp.items()}
    nt = -(-L // 128)
    # every query tile sees the sampled key tiles, so the forward covers the whole document
    sel = dict(q_tiles={0: list(range(nt))}, k_tiles={0: [0, nt - 1]}, bwd_q_tiles={0: [0, nt - 1]})
    o = run_oracle(sub, [L], gsz, 1, w.d, opts=O.Options(window=w.window), **sel)
    rows = np.r_[0:128, (nt - 1) * 128:L]
    gl = {key: (g[key][s0:s1][:, heads] if key in ("o", "dq") else g[key][s0:s1][:, [hk]]) for key in
          ("o", "dq", "dk", "dv")}
    for key in ("o", "dq", "dk", "dv"):
        e = norm_max_err(gl[key][rows], o[key][rows])
        assert e <= TOL, f"{key}: {e:.3e} cos {cosine(gl[key][rows], o[key][rows]):.6f}"
    lse_g = g["lse"][heads][:, s0:s1][:, rows]
    assert np.max(np.abs(lse_g - o["lse"][:, rows])) < 1e-3


def test_noncausal_documents_are_isolated_on_gpu():
    """Another document's inputs do not change this document's O, LSE, dK and dV
    bit for bit in a noncausal call (every quantity stays document-local)."""
    lengths, hq, hkv, d = [333, 400], 2, 2, 128
    inp = W.make_inputs(W.custom(lengths, hq, hkv, d, seed=32))
    a = run_gpu(inp, lengths, hq, hkv, d, window=(-1, -1))
    pert = {k_: v_.copy() for k_, v_ in inp.items()}
    for n in pert:
        pert[n][:333] = W.f32_to_bf16_bits(W.bf16_bits_to_f32(pert[n][:333]) * 8.0)
    b = run_gpu(pert, lengths, hq, hkv, d, window=(-1, -1))
    s = slice(333, 733)
    assert np.array_equal(a["o"][s], b["o"][s]) and np.array_equal(a["lse"][:, s], b["lse"][:, s])
    assert np.array_equal(a["dk"][s], b["dk"][s]) and np.array_equal(a["dv"][s], b["dv"][s])
