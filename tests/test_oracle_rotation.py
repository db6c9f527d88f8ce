"""Pins for the oracle's Hadamard rotation of Q and K (CPU only).

FLAMIA review section 3, "Rotation, range, and the alternative": an orthogonal
normalized Hadamard matrix rotates the head dimension before rounding, the
exact score is unchanged, and an isolated outlier is spread over every feature,
which helps a single coarse scale set by the largest entry; Korean review
section 3.4: the rotation is fused into the quantizer and is on by default at
head dim 128, and mixing channels within a token creates no causal dependency.
"""
import numpy as np
import pytest
import scipy.linalg

import oracle as O
from metrics import cosine


def _inputs(lengths, hq, hkv, d, seed=0, outliers=False):
    rng = np.random.default_rng(seed)
    T = int(sum(lengths))
    def mk(h):
        x = rng.standard_normal((T, h, d))
        if outliers:
            idx = rng.choice(x.size, size=max(1, x.size // 1000), replace=False)
            x.reshape(-1)[idx] *= 100.0
        return O.bf16_round(x)
    q, k, v, do = mk(hq), mk(hkv), mk(hkv), mk(hq)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(int)
    return q, k, v, do, cu


@pytest.mark.parametrize("d", [16, 64, 128])
def test_network_is_the_scaled_sylvester_hadamard_matrix(d):
    k = O.hadamard_norm_log2(d)
    assert 4 ** k >= d > 4 ** (k - 1)
    M = O.hadamard_rotate(np.eye(d), np.float64)          # row i = e_i H~
    assert np.array_equal(M, scipy.linalg.hadamard(d) / 2.0 ** k)
    assert np.array_equal(M, M.T)
    assert np.array_equal(M @ M, (d / 4.0 ** k) * np.eye(d))


def test_fp32_network_is_within_its_rounding_bound():
    """fp32 butterflies against the exact product: each output is a sum of d
    terms formed in log2(d) rounded stages, so |err| <= log2(d) 2^-24 sum|x| 2^-k."""
    rng = np.random.default_rng(1)
    d = 128
    x = O.bf16_round(rng.standard_normal((500, d)) * np.exp2(rng.integers(-8, 8, (500, 1))))
    exact = x @ scipy.linalg.hadamard(d) / 16.0
    got = O.hadamard_rotate(x, np.float32)
    bound = 7 * 2.0 ** -24 * np.abs(x).sum(-1, keepdims=True) / 16.0
    assert np.all(np.abs(got - exact) <= bound)
    assert not np.array_equal(got, exact)                  # it is not computed in fp64


@pytest.mark.parametrize("window", [(-1, 0), (-1, -1)])
def test_unquantized_rotated_attention_equals_unrotated(window):
    """The exact score is unchanged, so without quantization the rotated call
    (score scale times d / 4^k, dQ and dK rotated back) gives the same O, LSE and
    gradients."""
    lengths, hq, hkv = [300, 77, 129], 4, 2
    for d in (64, 128):
        q, k, v, do, cu = _inputs(lengths, hq, hkv, d, seed=2)
        base = O.run_training_call(q, k, v, do, cu, hq, hkv, opts=O.Options(quantized=False, window=window))
        rot = O.run_training_call(q, k, v, do, cu, hq, hkv,
                                  opts=O.Options(quantized=False, window=window, rotate=True))
        for n in ("o", "lse", "dq", "dk", "dv"):
            ref = base[n][np.isfinite(base[n])]
            got = rot[n][np.isfinite(base[n])]
            assert np.max(np.abs(got - ref)) <= 1e-11 * np.max(np.abs(ref)), (d, n)


def test_rotated_quantized_call_tracks_unquantized_attention():
    lengths, hq, hkv, d = [300, 200], 4, 2, 128
    q, k, v, do, cu = _inputs(lengths, hq, hkv, d, seed=3)
    out = O.run_training_call(q, k, v, do, cu, hq, hkv, opts=O.Options(rotate=True))
    ref_o, _ = O.dense_attention(q, k, v, cu, hq, hkv)
    ref_g = O.dense_attention_grads(q, k, v, do, cu, hq, hkv)
    assert cosine(out["o"], ref_o) > 0.997
    for n in ("dq", "dk", "dv"):
        assert cosine(out[n], ref_g[n]) > 0.99, n


def test_rotation_spreads_an_outlier_and_lowers_the_block_exponent():
    """One feature of one token 100x larger than the rest: unrotated, the block
    exponent follows the outlier; rotated, the outlier is spread over all 128
    features at about 1/sqrt(128) of its size, the exponent drops, and fewer of
    the block's small values fall below the E4M3 normal range."""
    rng = np.random.default_rng(4)
    x = O.bf16_round(rng.standard_normal((32, 1, 128)))
    x[5, 0, 17] = 400.0
    c0, s0 = O.quantize_tokenblock(x, [0, 32])
    xr = O.hadamard_rotate(x, np.float32)
    c1, s1 = O.quantize_tokenblock(xr, [0, 32])
    e0, e1 = int(s0[0, 0]) - 127, int(s1[0, 0]) - 127
    assert e1 < e0
    sub = lambda c: int(((c & 0x78) == 0).sum())            # zero or subnormal codes
    assert sub(c1) < sub(c0)
    # and the rotated reconstruction, rotated back, is closer to the input
    back = O.hadamard_rotate(O.dequantize_tokenblock(c1, s1), np.float64) * (4.0 ** 4 / 128)
    assert np.linalg.norm(back - x) < np.linalg.norm(O.dequantize_tokenblock(c0, s0) - x)


def test_rotated_call_on_outlier_inputs_still_tracks_unquantized_attention():
    """On inputs with 0.1% of entries 100x larger (the mixed-route workload's
    outliers) the rotated MXFP8 call still tracks unquantized attention.  The
    rotation does not help here: it drowns the other features of every token that
    holds an outlier, the trade-off the review names for fine scales; the measured
    cosines are recorded in the design notes."""
    lengths, hq, hkv, d = [256, 256], 2, 2, 128
    q, k, v, do, cu = _inputs(lengths, hq, hkv, d, seed=5, outliers=True)
    ref_o, _ = O.dense_attention(q, k, v, cu, hq, hkv)
    rot = O.run_training_call(q, k, v, do, cu, hq, hkv, opts=O.Options(rotate=True))
    assert cosine(rot["o"], ref_o) > 0.98


def test_rotation_keeps_earlier_blocks_bit_identical():
    """Mixing channels within a token consults no other position: a later 32-token
    block's perturbation leaves earlier rows' O and LSE bit-identical."""
    lengths, hq, hkv, d = [200], 2, 1, 64
    q, k, v, do, cu = _inputs(lengths, hq, hkv, d, seed=6)
    opts = O.Options(rotate=True)
    base = O.run_training_call(q, k, v, do, cu, hq, hkv, opts=opts)
    for name in ("q", "k", "v"):
        x = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
        x[name][133, 0, 7] *= 16.0
        pert = O.run_training_call(x["q"], x["k"], x["v"], do, cu, hq, hkv, opts=opts)
        assert np.array_equal(pert["o"][:128], base["o"][:128]), name
        assert np.array_equal(pert["lse"][:, :128], base["lse"][:, :128]), name


def test_planted_mistakes_fail_the_unquantized_equality():
    """Without the score-scale factor, or without rotating dQ and dK back, the
    unquantized rotated call no longer equals the unrotated one."""
    lengths, hq, hkv, d = [150], 2, 2, 128
    q, k, v, do, cu = _inputs(lengths, hq, hkv, d, seed=7)
    unq = O.Options(quantized=False)
    base = O.run_training_call(q, k, v, do, cu, hq, hkv, opts=unq)
    qr, kr = O.hadamard_rotate(q, np.float64), O.hadamard_rotate(k, np.float64)
    no_scale = O.run_training_call(qr, kr, v, do, cu, hq, hkv, opts=unq)          # scale not adjusted
    assert np.max(np.abs(no_scale["o"] - base["o"])) > 1e-3
    s = 1.0 / np.sqrt(d) * 2.0                                                      # scale adjusted, no rotate-back
    no_back = O.run_training_call(qr, kr, v, do, cu, hq, hkv, scale=s, opts=unq)
    assert np.max(np.abs(no_back["o"] - base["o"])) < 1e-12
    assert np.max(np.abs(no_back["dq"] - base["dq"])) > 1e-3
