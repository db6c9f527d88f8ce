"""GPU parity of the Hadamard-rotated calls against the oracle.

FLAMIA review section 3, "Rotation, range, and the alternative"; Korean review
section 3.4 (rotation fused into the quantizer, on by default at head dim 128).
Q and K are rotated per token by H / 2^k in fp32 before quantization, so their
codes, scale bytes and row statistics are bit-exact with the oracle; O, LSE and
the gradients (dQ, dK rotated back) are within the usual bar.
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
    ("causal_ragged_gqa_d128", [300, 77, 129, 1], 4, 2, 128, 5, (-1, 0), "normal"),
    ("causal_d64", [256, 130], 2, 2, 64, 0, (-1, 0), "normal"),
    ("noncausal_d128", [333, 200], 2, 1, 128, 0, (-1, -1), "normal"),
    ("outliers_d128", [400, 112], 2, 2, 128, 0, (-1, 0), "normal_outliers"),
    ("student_t_d128", [700], 2, 1, 128, 3, (-1, 0), "student_t3"),
]


@pytest.mark.parametrize("name,lengths,hq,hkv,d,extra,window,dist", CASES, ids=[c[0] for c in CASES])
def test_rotated_training_call_matches_oracle(name, lengths, hq, hkv, d, extra, window, dist):
    T = sum(lengths) + extra
    inp = W.make_inputs(W.custom([T], hq, hkv, d, dist=dist, seed=41))
    g = run_gpu(inp, lengths, hq, hkv, d, total_tokens=T, window=window, rotate=True)
    o = run_oracle(inp, lengths, hq, hkv, d, opts=O.Options(window=window, rotate=True))
    assert g["status"] == 0
    for n in ("q", "k", "v"):
        assert np.array_equal(g[n + "_codes"], o[n + "_codes"]), n
        assert np.array_equal(g[n + "_scales"], o[n + "_scales"]), n
    valid = sum(lengths)
    # K row statistics of the rotated codes (they feed the dQ boost)
    kh = o["k_hat"][:valid]
    assert np.allclose(g["k_stats"][:valid, :, 0], np.sqrt((kh ** 2).sum(-1)), rtol=1e-5)
    assert np.array_equal(g["k_stats"][:valid, :, 1], np.abs(kh).max(-1).astype(np.float32))
    assert np.max(np.abs(g["lse"][:, :valid] - o["lse"][:, :valid])) < 1e-3
    for n in ("o", "dq", "dk", "dv"):
        e = norm_max_err(g[n], o[n])
        assert e <= TOL, f"{n}: {e:.3e} cos {cosine(g[n], o[n]):.6f}"
        assert np.all(g[n][valid:] == 0), n


def test_rotated_gpu_call_tracks_unquantized_attention_like_the_oracle():
    lengths, hq, hkv, d = [700, 324], 4, 2, 128
    inp = W.make_inputs(W.custom([sum(lengths)], hq, hkv, d, seed=42))
    g = run_gpu(inp, lengths, hq, hkv, d, rotate=True)
    o = run_oracle(inp, lengths, hq, hkv, d, opts=O.Options(rotate=True))
    vals = {n: W.bf16_bits_to_f32(inp[n]).astype(np.float64) for n in inp}
    cu = np.concatenate([[0], np.cumsum(lengths)])
    ref_o, _ = O.dense_attention(vals["q"], vals["k"], vals["v"], cu, hq, hkv)
    ref_g = O.dense_attention_grads(vals["q"], vals["k"], vals["v"], vals["do"], cu, hq, hkv)
    co_g, co_o = cosine(g["o"], ref_o), cosine(o["o"], ref_o)
    assert co_g > 0.998 and abs(co_g - co_o) < 2e-4, (co_g, co_o)
    for n in ("dq", "dk", "dv"):
        cg, cor = cosine(g[n], ref_g[n]), cosine(o[n], ref_g[n])
        assert cg > 0.995 and abs(cg - cor) < 5e-4, (n, cg, cor)
