"""GPU parity of the causal MXFP8 forward and backward against the oracle.

Tolerance: O, dQ, dK and dV within 1e-2 of the oracle in max-abs error
normalised by the oracle tensor's max-abs (the two sides round the same E4M3
operands but accumulate in different orders, and ex2.approx differs from the
oracle's fp64 exponential by a few fp32 ulps, which can move an E4M3 rounding by
one code); codes and scale bytes bit-exact; LSE within 1e-3 absolute (natural
log).
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


def _compare(g, o, names=("o", "dq", "dk", "dv"), rows=None, heads=None, kv_heads=None):
    msgs, worst = [], 0.0
    for n in names:
        a, b = g[n], o[n]
        if rows is not None:
            a, b = a[rows], b[rows]
        hs = kv_heads if n in ("dk", "dv") else heads
        if hs is not None:
            a, b = a[:, hs], b[:, hs]
        e = norm_max_err(a, b)
        worst = max(worst, e)
        msgs.append(f"{n}: err {e:.2e} cos {cosine(a, b):.6f}")
    return worst, "; ".join(msgs)


CASES = [
    ("ragged_gqa_d128", [300, 77, 129, 1], 2, 1, 128, 0),
    ("batched_b1_h2_s256_d64", [256], 2, 2, 64, 0),
    ("gqa4_two_docs_d128", [200, 517], 4, 1, 128, 0),
    ("mha_tail_d64", [130, 5, 260], 2, 2, 64, 19),
]


@pytest.mark.parametrize("name,lengths,hq,hkv,d,extra", CASES, ids=[c[0] for c in CASES])
def test_training_call_matches_oracle(name, lengths, hq, hkv, d, extra):
    T = sum(lengths) + extra
    w = W.custom([T], hq, hkv, d, seed=7)
    inp = W.make_inputs(w)
    g = run_gpu(inp, lengths, hq, hkv, d, total_tokens=T)
    o = run_oracle(inp, lengths, hq, hkv, d)
    assert g["status"] == 0
    for n in ("q", "k", "v"):
        assert np.array_equal(g[n + "_codes"], o[n + "_codes"]), n
        assert np.array_equal(g[n + "_scales"], o[n + "_scales"]), n
    assert np.array_equal(g["do_codes"], o["do_codes"]) and np.array_equal(g["do_scales"], o["do_scales"])
    valid = sum(lengths)
    lse_err = np.max(np.abs(g["lse"][:, :valid] - o["lse"][:, :valid]))
    assert lse_err < 1e-3, lse_err
    assert np.all(np.isinf(g["lse"][:, valid:])) and np.all(g["o"][valid:] == 0)
    worst, msg = _compare(g, o)
    assert worst <= TOL, msg
    for n in ("dq", "dk", "dv"):
        assert np.all(g[n][valid:] == 0), n


def test_forward_is_deterministic_and_prefix_isolated():
    """Bitwise: two runs agree; a perturbation in a later 32-token block leaves
    O and LSE of earlier rows unchanged (suffix test, FLAMIA review section 10)."""
    lengths, hq, hkv, d = [700], 2, 1, 128
    w = W.custom(lengths, hq, hkv, d, seed=9)
    inp = W.make_inputs(w)
    a = run_gpu(inp, lengths, hq, hkv, d, with_bwd=False)
    b = run_gpu(inp, lengths, hq, hkv, d, with_bwd=False)
    assert np.array_equal(a["o"], b["o"]) and np.array_equal(a["lse"], b["lse"])
    blk = 13                                           # tokens 416..447
    for name in ("q", "k", "v"):
        pert = {k_: v_.copy() for k_, v_ in inp.items()}
        x = W.bf16_bits_to_f32(pert[name][blk * 32 + 5, 0, 3:4]) * 16.0
        pert[name][blk * 32 + 5, 0, 3:4] = W.f32_to_bf16_bits(x)
        c = run_gpu(pert, lengths, hq, hkv, d, with_bwd=False)
        lim = blk * 32
        assert np.array_equal(c["o"][:lim], a["o"][:lim]), name
        assert np.array_equal(c["lse"][:, :lim], a["lse"][:, :lim]), name


def test_documents_are_isolated_on_gpu():
    """Negative control: another document's inputs do not change this document's
    O, LSE, dK, dV bit for bit (dQ is reduced with atomics in any order)."""
    lengths, hq, hkv, d = [333, 400], 2, 2, 128
    w = W.custom(lengths, hq, hkv, d, seed=12)
    inp = W.make_inputs(w)
    a = run_gpu(inp, lengths, hq, hkv, d)
    pert = {k_: v_.copy() for k_, v_ in inp.items()}
    for n in pert:
        pert[n][:333] = W.f32_to_bf16_bits(W.bf16_bits_to_f32(pert[n][:333]) * 8.0)
    b = run_gpu(pert, lengths, hq, hkv, d)
    s = slice(333, 733)
    assert np.array_equal(a["o"][s], b["o"][s]) and np.array_equal(a["lse"][:, s], b["lse"][:, s])
    assert np.array_equal(a["dk"][s], b["dk"][s]) and np.array_equal(a["dv"][s], b["dv"][s])
    assert norm_max_err(b["dq"][s], a["dq"][s]) < 1e-2


@pytest.mark.parametrize("wname", ["packed_16k_h16_d128", "gqa_b4_s8192_hq32_hkv8_d128", "skewed_8192_224x256_h16_d128"])
def test_full_size_sampled_parity(wname):
    """The full workload on the GPU in the benchmark's launch configuration; the
    oracle recomputes one document x one kv-head group on sampled tiles."""
    w = W.WORKLOADS[wname]
    inp = W.make_inputs(w)
    g = run_gpu(inp, list(w.lengths), w.hq, w.hkv, w.d)
    assert g["status"] == 0
    lengths = list(w.lengths)
    n = int(np.argmax(lengths))                       # the longest document
    s0 = int(np.sum(lengths[:n])); L = lengths[n]; s1 = s0 + L
    hk = w.hkv - 1
    gsz = w.hq // w.hkv
    heads = list(range(hk * gsz, (hk + 1) * gsz))
    sub = {name: arr[s0:s1][:, heads if name in ("q", "do") else [hk]] for name, arr in inp.items()}
    nt = -(-L // 128)
    sel = dict(q_tiles={0: [0, nt - 2, nt - 1]}, k_tiles={0: [nt - 2, nt - 1]}, bwd_q_tiles={0: [0, nt - 1]})
    o = run_oracle(sub, [L], gsz, 1, w.d, **sel)
    rows_o = np.r_[0:128, (nt - 2) * 128:L]
    rows_q = np.r_[0:128, (nt - 1) * 128:L]
    rows_k = np.r_[(nt - 2) * 128:L]
    gl = {key: (g[key][s0:s1][:, heads] if key in ("o", "dq") else g[key][s0:s1][:, [hk]]) for key in
          ("o", "dq", "dk", "dv")}
    for key, rows in (("o", rows_o), ("dq", rows_q), ("dk", rows_k), ("dv", rows_k)):
        e = norm_max_err(gl[key][rows], o[key][rows])
        assert e <= TOL, f"{key}: {e:.3e} cos {cosine(gl[key][rows], o[key][rows]):.6f}"
    lse_g = g["lse"][heads][:, s0:s1][:, rows_o]
    assert np.max(np.abs(lse_g - o["lse"][:, rows_o])) < 1e-3
    for nme in ("q", "k", "v"):
        hsel = heads if nme == "q" else [hk]
        assert np.array_equal(g[nme + "_codes"][s0:s1][:, hsel], o[nme + "_codes"]), nme


EDGE_CASES = [
    # empty documents in the middle and at the end, one-token documents, a document
    # of exactly one 128-token tile and one of exactly one 32-token block
    ("empty_and_tiny_docs", [0, 37, 0, 1, 128, 32, 1, 0], 2, 1, 128, 5),
    # wide GQA group (8 query heads per kv head) across tile boundaries
    ("gqa8_ragged", [129, 255, 256], 8, 1, 64, 0),
    # MHA with many heads, lengths just past the 32-token block and 128-token tile sizes
    ("mha_h6_boundaries", [33, 129, 161, 97], 6, 6, 128, 3),
]


@pytest.mark.parametrize("name,lengths,hq,hkv,d,extra", EDGE_CASES, ids=[c[0] for c in EDGE_CASES])
def test_edge_layouts_match_oracle(name, lengths, hq, hkv, d, extra):
    T = sum(lengths) + extra
    w = W.custom([T], hq, hkv, d, seed=17)
    inp = W.make_inputs(w)
    g = run_gpu(inp, lengths, hq, hkv, d, total_tokens=T)
    o = run_oracle(inp, lengths, hq, hkv, d)
    assert g["status"] == 0
    for n in ("q", "k", "v"):
        assert np.array_equal(g[n + "_codes"], o[n + "_codes"]), n
        assert np.array_equal(g[n + "_scales"], o[n + "_scales"]), n
    valid = sum(lengths)
    assert np.max(np.abs(g["lse"][:, :valid] - o["lse"][:, :valid])) < 1e-3
    worst, msg = _compare(g, o)
    assert worst <= TOL, msg
    for n in ("o", "dq", "dk", "dv"):
        assert np.all(g[n][valid:] == 0), n


def test_gpu_tracks_unquantized_attention_like_the_oracle():
    """The cosine against unquantized fp64 attention (the pages report 0.9988 for
    the output and 0.9979 for the gradients of the MXFP8 route, [EN] section 8):
    the GPU lands where the oracle does, so the gap to 0.999 on gradients is the
    E4M3 rounding of the method, not the kernels (risk R1 in the design notes)."""
    lengths, hq, hkv, d = [700, 324], 4, 2, 128
    w = W.custom([sum(lengths)], hq, hkv, d, seed=18)
    inp = W.make_inputs(w)
    g = run_gpu(inp, lengths, hq, hkv, d)
    o = run_oracle(inp, lengths, hq, hkv, d)
    vals = {n: W.bf16_bits_to_f32(inp[n]).astype(np.float64) for n in inp}
    cu = np.concatenate([[0], np.cumsum(lengths)])
    ref_o, _ = O.dense_attention(vals["q"], vals["k"], vals["v"], cu, hq, hkv)
    ref_g = O.dense_attention_grads(vals["q"], vals["k"], vals["v"], vals["do"], cu, hq, hkv)
    co_g, co_o = cosine(g["o"], ref_o), cosine(o["o"], ref_o)
    assert co_g > 0.998 and abs(co_g - co_o) < 2e-4, (co_g, co_o)
    for n in ("dq", "dk", "dv"):
        cg, cor = cosine(g[n], ref_g[n]), cosine(o[n], ref_g[n])
        assert cg > 0.995 and abs(cg - cor) < 5e-4, (n, cg, cor)


def test_training_call_replays_from_a_cuda_graph():
    """The calls need no host synchronisation and allocate nothing, so the whole
    training call (plan, quantize, forward, backward) can be captured into one CUDA
    graph ([EN] section 6: graph-capturable, row capacity independent of the
    document lengths). Replays match the eager call (dQ up to the order of its
    fp16 reductions)."""
    import torch
    import microscaled_precision_causal_gb300 as F
    from gpu_harness import to_device_bf16, cu_tensor
    lengths, hq, hkv, d = [300, 77, 129], 4, 2, 128
    T = sum(lengths) + 7
    inp = W.make_inputs(W.custom([T], hq, hkv, d, seed=19))
    x = {n: to_device_bf16(inp[n]) for n in inp}
    cu = cu_tensor(lengths)
    att = F.FlamiaAttention(T, len(lengths), hq, hkv, d)
    att.training_call(x["q"], x["k"], x["v"], x["do"], cu)
    torch.cuda.synchronize()
    eager = {n: getattr(att, n).clone() for n in ("out", "lse", "dq", "dk", "dv")}
    for t in (att.out, att.dq, att.dk, att.dv):
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        att.training_call(x["q"], x["k"], x["v"], x["do"], cu)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert att.device_status() == 0
    for n in ("out", "lse", "dk", "dv"):
        assert torch.equal(getattr(att, n), eager[n]), n
    a, b = att.dq.float().cpu().numpy(), eager["dq"].float().cpu().numpy()
    assert norm_max_err(a, b) < 2e-3


@pytest.mark.gpu
def test_forward_document_longer_than_the_scale_table():
    """A document of more than 1024 key tiles (131,972 tokens): each forward softmax
    warpgroup stages the K/V scale bytes of at most 1024 key tiles in shared memory and
    reads those of later tiles from global memory; the last query tiles use both, the
    first tile only the table.  O and LSE of those tiles against the oracle."""
    L = 1024 * 128 + 900
    lengths = [300, L]
    w = W.Workload("long_document", tuple(lengths), 1, 1, 64, seed=11)
    inp = W.make_inputs(w, tensors=("q", "k", "v"))
    g = run_gpu(inp, lengths, 1, 1, 64, with_bwd=False)
    assert g["status"] == 0
    s0 = lengths[0]
    sub = {n: inp[n][s0:s0 + L] for n in ("q", "k", "v")}
    nt = -(-L // 128)
    o = run_oracle(sub, [L], 1, 1, 64, with_bwd=False, q_tiles={0: [0, nt - 2, nt - 1]})
    rows = np.r_[0:128, (nt - 2) * 128:L]
    e = norm_max_err(g["o"][s0:s0 + L][rows], o["o"][rows])
    assert e <= TOL, f"o: {e:.3e}"
    assert np.max(np.abs(g["lse"][:, s0:s0 + L][:, rows] - o["lse"][:, rows])) < 1e-3
