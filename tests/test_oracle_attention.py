"""Pins for the oracle's attention, cost model and work list (CPU only)."""
import math

import numpy as np
import pytest

import oracle as O
from golden_io import rows
from metrics import cosine, norm_max_err


def _inputs(lengths, hq, hkv, d, seed=0, scale=1.0, bf16=True):
    rng = np.random.default_rng(seed)
    T = int(sum(lengths))
    mk = lambda h: rng.standard_normal((T, h, d)) * scale
    q, k, v, do = mk(hq), mk(hkv), mk(hkv), mk(hq)
    if bf16:
        q, k, v, do = (O.bf16_round(x) for x in (q, k, v, do))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(int)
    return q, k, v, do, cu


# ------------------------------------------------------------ cost model

def _parse_lengths(spec):
    out = []
    for part in spec.split("+"):
        n, L = part.split("x")
        out += [int(L)] * int(n)
    return out


def test_visible_pairs_from_pages():
    for spec, pairs in rows("pair_counts.txt"):
        L = _parse_lengths(spec)
        assert sum(L) == 65536
        assert O.visible_pairs(L) == int(pairs)


def test_visible_pairs_brute_force():
    for L in ([1], [5, 3], [17, 1, 2, 40]):
        cu = np.concatenate([[0], np.cumsum(L)])
        brute = sum(1 for s, t in O.doc_ranges(cu) for i in range(s, t) for j in range(s, t) if j <= i)
        assert O.visible_pairs(L) == brute


# ------------------------------------------------------------ unquantized attention

UNQ = O.Options(quantized=False)


@pytest.mark.parametrize("lengths,hq,hkv,d", [([300, 77, 129, 1], 2, 1, 16), ([256], 2, 2, 8), ([130, 5], 4, 2, 8)])
def test_tiled_forward_equals_dense_bruteforce(lengths, hq, hkv, d):
    q, k, v, do, cu = _inputs(lengths, hq, hkv, d)
    O1, L1 = O.attention_forward(q, k, v, cu, hq, hkv, opts=UNQ)
    O2, L2 = O.dense_attention(q, k, v, cu, hq, hkv)
    assert np.max(np.abs(O1 - O2)) <= 1e-12 * np.max(np.abs(O2))
    assert np.max(np.abs(L1 - L2)) <= 1e-12 * np.max(np.abs(L2))


def test_online_softmax_is_block_partition_invariant():
    """[FA] "Attention without the score matrix": blocks of 32 keys agree with ordinary attention."""
    q, k, v, do, cu = _inputs([200, 64], 2, 2, 8, seed=1)
    ref, _ = O.dense_attention(q, k, v, cu, 2, 2)
    for tile in (32, 64, 128):
        o, _ = O.attention_forward(q, k, v, cu, 2, 2, opts=O.Options(quantized=False, tile=tile))
        assert np.max(np.abs(o - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_dense_gradients_match_finite_differences():
    """Autograd-free central differences of L = sum(dO * O) on tiny shapes."""
    lengths, hq, hkv, d = [7, 5], 2, 1, 4
    q, k, v, do, cu = _inputs(lengths, hq, hkv, d, seed=2, bf16=False)
    g = O.dense_attention_grads(q, k, v, do, cu, hq, hkv)
    loss = lambda q_, k_, v_: float((O.dense_attention(q_, k_, v_, cu, hq, hkv)[0] * do).sum())
    eps = 1e-6
    for name, x, gx in (("q", q, g["dq"]), ("k", k, g["dk"]), ("v", v, g["dv"])):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp = x.copy(); xp[idx] += eps
            xm = x.copy(); xm[idx] -= eps
            args = {"q": q, "k": k, "v": v}
            args[name] = xp; lp = loss(args["q"], args["k"], args["v"])
            args[name] = xm; lm = loss(args["q"], args["k"], args["v"])
            num[idx] = (lp - lm) / (2 * eps)
        assert np.max(np.abs(num - gx)) <= 1e-6 * max(1.0, np.max(np.abs(gx))), name


@pytest.mark.parametrize("lengths,hq,hkv,d", [([300, 77, 129, 1], 2, 1, 16), ([140, 33], 4, 2, 8)])
def test_tiled_backward_equals_dense_gradients(lengths, hq, hkv, d):
    q, k, v, do, cu = _inputs(lengths, hq, hkv, d, seed=3)
    o, lse = O.attention_forward(q, k, v, cu, hq, hkv, opts=UNQ)
    gt = O.attention_backward(q, k, v, o, lse, do, cu, hq, hkv, opts=UNQ)
    gd = O.dense_attention_grads(q, k, v, do, cu, hq, hkv)
    for n in ("dq", "dk", "dv"):
        assert np.max(np.abs(gt[n] - gd[n])) <= 1e-11 * np.max(np.abs(gd[n])), n


def test_centered_softmax_gradient_row_invariant():
    """[EN] section 2: sum_j dS_ij = 0 with matched P and normalisation."""
    q, k, v, do, cu = _inputs([250, 40], 2, 2, 16, seed=4)
    o, lse = O.attention_forward(q, k, v, cu, 2, 2, opts=UNQ)
    g = O.attention_backward(q, k, v, o, lse, do, cu, 2, 2, opts=UNQ, diagnostics=True)
    rs, rm = g["diag"]["rowsum_ds"], g["diag"]["rowmax_ds"]
    assert np.max(np.abs(rs) / np.maximum(rm, 1e-300)) < 1e-12
    assert np.max(np.abs(O.dense_attention_grads(q, k, v, do, cu, 2, 2)["ds_rowsum"])) < 1e-12


# ------------------------------------------------------------ quantized path properties

def test_quantized_path_tracks_unquantized_attention():
    """The pages report cosines near 0.999 (output) and 0.998 (gradients) for MXFP8
    against an FP32 reference ([EN] section 8); a dropped term, transposed operand or
    wrong sign in the quantized oracle would fall far below these loose bounds."""
    lengths, hq, hkv, d = [300, 200], 4, 2, 64
    q, k, v, do, cu = _inputs(lengths, hq, hkv, d, seed=5)
    out = O.run_training_call(q, k, v, do, cu, hq, hkv)
    ref_o, _ = O.dense_attention(q, k, v, cu, hq, hkv)
    ref_g = O.dense_attention_grads(q, k, v, do, cu, hq, hkv)
    assert cosine(out["o"], ref_o) > 0.997
    for n in ("dq", "dk", "dv"):
        assert cosine(out[n], ref_g[n]) > 0.99, n
        assert norm_max_err(out[n], ref_g[n]) < 0.15, n


def test_forward_p_quantization_bound():
    """With tau = 0 every boosted weight is <= 2**8 and never clips ([EN] section 5)."""
    q, k, v, do, cu = _inputs([130], 1, 1, 16, seed=6, scale=3.0)
    o0, _ = O.attention_forward(q, k, v, cu, 1, 1, opts=O.Options(p_boost_log2=8))
    # the same call with beta = 2**8 and an unclipped codec differs only by rounding
    o1, _ = O.attention_forward(q, k, v, cu, 1, 1, opts=O.Options(quantized=False))
    assert cosine(o0, o1) > 0.999


def test_lagging_max_with_tempting_boost_clips():
    """[EN] section 5: tau = 2, beta = 2**8 lets a weight of 4 clip to 448/256 = 1.75."""
    d = 2
    # one query; key tile 0 holds a score of 0, key tile 1 a score of ln(4) (= 2 in log2 units)
    T = 129
    q = np.zeros((T, 1, d)); k = np.zeros((T, 1, d)); v = np.zeros((T, 1, d))
    q[128, 0, 0] = 1.0
    k[128, 0, 0] = math.log(4.0)                 # scale = 1 below
    v[128, 0, 1] = 1.0
    cu = [0, T]
    opts = O.Options(p_lag_log2=2, p_boost_log2=8, quantized=True)
    o, lse = O.attention_forward(q, k, v, cu, 1, 1, scale=1.0, opts=opts)
    # row 128: 128 keys with weight 1 (tile 0, retained max 0), one key with weight 4 -> 1.75
    assert o[128, 0, 1] == O.bf16_round(1.75 / (128 + 4.0))
    o_ok, _ = O.attention_forward(q, k, v, cu, 1, 1, scale=1.0, opts=O.Options())
    assert abs(o_ok[128, 0, 1] - 4.0 / 132.0) < 4.0 / 132.0 / 64


# ------------------------------------------------------------ prefix isolation

def _train(q, k, v, do, cu, hq, hkv, **kw):
    return O.run_training_call(q, k, v, do, cu, hq, hkv, opts=O.Options(**kw))


def test_suffix_perturbation_leaves_earlier_blocks_bit_identical():
    """[EN] section 10 / [KO] section 4.5: changing tokens in a later 32-token block
    leaves O and LSE of queries in earlier blocks bit-identical (default path)."""
    lengths, hq, hkv, d = [260], 2, 1, 32
    q, k, v, do, cu = _inputs(lengths, hq, hkv, d, seed=8)
    base = _train(q, k, v, do, cu, hq, hkv)
    bp = 5                                     # perturb block 5 = tokens 160..191
    for name in ("q", "k", "v"):
        x = {"q": q, "k": k, "v": v}
        y = x[name].copy()
        y[bp * 32 + 3, 0, 1] *= 16.0               # push the block amax over exponent thresholds
        x[name] = y
        pert = _train(x["q"], x["k"], x["v"], do, cu, hq, hkv)
        lim = bp * 32
        assert np.array_equal(pert["o"][:lim], base["o"][:lim]), name
        assert np.array_equal(pert["lse"][:, :lim], base["lse"][:, :lim]), name
        assert not np.array_equal(pert["o"], base["o"]) or name == "q"


def test_within_block_perturbation_is_detected():
    """Positive control: a later token inside the same 32-token block moves the
    block exponent and changes an earlier row's output (the residual in-block leak
    the pages describe for the default token-block scales)."""
    lengths, hq, hkv, d = [64], 1, 1, 16
    q, k, v, do, cu = _inputs(lengths, hq, hkv, d, seed=9)
    base = _train(q, k, v, do, cu, hq, hkv)
    v2 = v.copy(); v2[40, 0, 0] *= 2.0 ** 12        # same block as rows 32..63
    pert = _train(q, k, v2, do, cu, hq, hkv)
    assert np.array_equal(pert["o"][:32], base["o"][:32])
    assert not np.array_equal(pert["o"][32:40], base["o"][32:40])


def test_floor_rule_leaks_through_clamp_roundup_does_not():
    """The clamp mechanism of [KO] section 2: with the floor rule, a masked later
    token in the same block that lifts the amax across 448*2^k un-clips an
    earlier value; round-up keeps the reconstruction (normal codes)."""
    T, d = 32, 4
    v = np.ones((T, 1, d)) * 1.0
    v[3, 0, 0] = 460.0
    v2 = v.copy(); v2[20, 0, 1] = 900.0
    cu = [0, T]
    f1 = O.dequantize_tokenblock(*O.quantize_tokenblock(v, cu, rule="floor"))
    f2 = O.dequantize_tokenblock(*O.quantize_tokenblock(v2, cu, rule="floor"))
    assert f1[3, 0, 0] == 448.0 and f2[3, 0, 0] == 448.0        # clamp, then RNE of 230
    v[3, 0, 0] = 480.0; v2[3, 0, 0] = 480.0
    f1 = O.dequantize_tokenblock(*O.quantize_tokenblock(v, cu, rule="floor"))
    f2 = O.dequantize_tokenblock(*O.quantize_tokenblock(v2, cu, rule="floor"))
    assert f1[3, 0, 0] == 448.0 and f2[3, 0, 0] == 480.0        # the leak
    r1 = O.dequantize_tokenblock(*O.quantize_tokenblock(v, cu))
    r2 = O.dequantize_tokenblock(*O.quantize_tokenblock(v2, cu))
    assert r1[3, 0, 0] == r2[3, 0, 0] == 480.0


def test_documents_are_isolated_and_offset_invariant():
    """Negative control ([EN] section 10): another document's inputs and a
    document's physical offset do not change its outputs or gradients."""
    hq, hkv, d = 2, 1, 16
    q, k, v, do, cu = _inputs([150, 90], hq, hkv, d, seed=10)
    base = _train(q, k, v, do, cu, hq, hkv)
    s = slice(150, 240)
    q2 = q.copy(); q2[:150] *= 8; k2 = k.copy(); k2[:150] *= 0.25
    pert = _train(q2, k2, v, do, cu, hq, hkv)
    for n in ("o", "dq", "dk", "dv"):
        assert np.array_equal(pert[n][s], base[n][s]), n
    for shift in (1, 37, 127):
        rng = np.random.default_rng(shift)
        pre = lambda h: O.bf16_round(rng.standard_normal((shift, h, d)))
        qs = np.concatenate([pre(hq), q[s]]); ks = np.concatenate([pre(hkv), k[s]])
        vs = np.concatenate([pre(hkv), v[s]]); dos = np.concatenate([pre(hq), do[s]])
        out = _train(qs, ks, vs, dos, [0, shift, shift + 90], hq, hkv)
        for n in ("o", "dq", "dk", "dv"):
            assert np.array_equal(out[n][shift:], base[n][s]), (n, shift)


def test_dq_boost_definition():
    rng = np.random.default_rng(12)
    for _ in range(50):
        a = rng.standard_normal((20, 8)) * np.exp2(rng.integers(-20, 20))
        b = rng.standard_normal((20, 8)); c = rng.standard_normal((20, 8))
        M = 2 * np.linalg.norm(a, axis=1).max() * np.linalg.norm(b, axis=1).max() * np.abs(c).max()
        boost = O.dq_boost(a, b, c)
        e = math.log2(boost)
        assert e == int(e)
        assert boost * M <= 2 ** 14 < 2 * boost * M
    assert O.dq_boost(np.zeros((3, 4)), np.ones((3, 4)), np.ones((3, 4))) == 1.0


def test_dq_boost_keeps_fp16_partials_in_range():
    q, k, v, do, cu = _inputs([256], 1, 1, 32, seed=13, scale=20.0)
    out = O.run_training_call(q, k, v, do, cu, 1, 1)
    assert np.all(np.isfinite(out["dq"]))


# ------------------------------------------------------------ work list

def test_work_list_order_and_alternation():
    cu = [0, 1000, 1200, 1201, 5000]
    items = O.work_list(cu, num_ctas=3)
    costs = [it["cost"] for it in items]
    assert costs == sorted(costs, reverse=True)
    # every (doc, query tile) covered exactly once, items <= 256 queries
    seen = set()
    for it in items:
        assert 1 <= it["ntiles"] <= 2
        for t in range(it["tile0"], it["tile0"] + it["ntiles"]):
            assert (it["doc"], t) not in seen
            seen.add((it["doc"], t))
    want = {(n, t) for n, (s, e) in enumerate(O.doc_ranges(cu)) for t in range(-(-(e - s) // 128))}
    assert seen == want
    # cost = visible 128-key tiles summed over the item's query tiles
    for it in items:
        assert it["cost"] == sum(t + 1 for t in range(it["tile0"], it["tile0"] + it["ntiles"]))
    # boustrophedon: 0 1 2 | 2 1 0 | 0 1 2 ...
    assert [it["cta"] for it in items[:9]] == [0, 1, 2, 2, 1, 0, 0, 1, 2]
    # ties keep document order
    first_doc = [it["doc"] for it in items if it["cost"] == items[-1]["cost"]]
    assert first_doc == sorted(first_doc)


def test_bwd_key_tile_list():
    cu = [0, 300, 301, 700]        # 3, 1 and 4 key tiles
    items = O.bwd_key_tile_list(cu)
    got = [(i["doc"], i["ktile"], i["cost"]) for i in items]
    assert got == [(2, 0, 4), (0, 0, 3), (2, 1, 3), (0, 1, 2), (2, 2, 2),
                   (0, 2, 1), (1, 0, 1), (2, 3, 1)]


# ------------------------------------------------------------ strict options

def _strict(q, k, v, do, cu, hq, hkv):
    return O.run_training_call(q, k, v, do, cu, hq, hkv, opts=O.Options(strict=True))


def test_strict_options_make_earlier_rows_bit_identical():
    """[EN] section 4 / [KO] section 4.5: with per-token operand scales, per-row
    dS exponents and the causal dQ scale, perturbing any later token (with dO
    fixed) leaves O, LSE and dQ of every earlier row bit-identical."""
    lengths, hq, hkv, d = [290, 60], 2, 1, 32
    rng = np.random.default_rng(20)
    T = sum(lengths)
    mk = lambda h: O.bf16_round(rng.standard_t(3, (T, h, d)))
    q, k, v, do = mk(hq), mk(hkv), mk(hkv), mk(hq)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    base = _strict(q, k, v, do, cu, hq, hkv)
    for t in (1, 33, 150, 289):
        for name in ("q", "k", "v"):
            x = {"q": q, "k": k, "v": v}
            y = x[name].copy()
            y[t] *= 16.0                                   # crosses exponent thresholds
            x[name] = y
            pert = _strict(x["q"], x["k"], x["v"], do, cu, hq, hkv)
            assert np.array_equal(pert["o"][:t], base["o"][:t]), (name, t)
            assert np.array_equal(pert["lse"][:, :t], base["lse"][:, :t]), (name, t)
            assert np.array_equal(pert["dq"][:t], base["dq"][:t]), (name, t)
            if name != "q":   # positive control: the perturbed key/value reaches its own row
                assert not np.array_equal(pert["o"][t], base["o"][t]), (name, t)


def test_default_dq_boost_leaks_across_the_sequence():
    """Negative counterpart: the default sequence-wide dQ boost lets a later
    outlier change earlier dQ rows (the residual dependency the pages report)."""
    lengths, hq, hkv, d = [200], 1, 1, 16
    q, k, v, do, cu = _inputs(lengths, hq, hkv, d, seed=21)
    base = O.run_training_call(q, k, v, do, cu, hq, hkv)
    do2 = do.copy(); do2[190] *= 2.0 ** 20                 # lowers the sequence-wide boost by ~2^20
    pert = O.run_training_call(q, k, v, do2, cu, hq, hkv)
    # earlier rows' fp16 partials now round at a coarser relative step
    assert not np.array_equal(pert["dq"][:128], base["dq"][:128])
    strict_b = O.run_training_call(q, k, v, do, cu, hq, hkv, opts=O.Options(strict=True))
    strict_p = O.run_training_call(q, k, v, do2, cu, hq, hkv, opts=O.Options(strict=True))
    assert np.array_equal(strict_p["dq"][:190], strict_b["dq"][:190])


def test_fold_quantize_roundup_groups():
    rng = np.random.default_rng(22)
    X = rng.standard_normal((40, 70)) * np.exp2(rng.integers(-10, 10, (40, 70)))
    R = O.flamia_oracle._fold_quantize(X, group_axis=1, offset=0)
    for g0 in range(0, 70, 32):
        blk = X[:, g0:g0 + 32]
        e = O.roundup_exponent(np.abs(blk).max(1))
        want = O.e4m3_round(blk * np.exp2(-e)[:, None]) * np.exp2(e)[:, None]
        assert np.array_equal(R[:, g0:g0 + 32], want)
        scaled = np.abs(blk).max(1) * np.exp2(-e.astype(float))
        assert np.all((scaled > 224) & (scaled <= 448))
    R0 = O.flamia_oracle._fold_quantize(X.T, group_axis=0, offset=32)
    assert np.array_equal(R0, R.T)


def test_causal_dq_boost_is_prefix_local():
    rng = np.random.default_rng(23)
    a, b, c = rng.standard_normal((50, 8)), rng.standard_normal((50, 8)), rng.standard_normal((50, 8))
    full = O.causal_dq_boost(a, b, c)
    for i in (0, 7, 31, 49):
        M = 2 * np.linalg.norm(a[i]) * np.linalg.norm(b[:i + 1], axis=1).max() * np.abs(c[:i + 1]).max()
        assert full[i] * M <= 2 ** 14 < 2 * full[i] * M
        assert O.causal_dq_boost(a[:i + 1], b[:i + 1], c[:i + 1])[i] == full[i]


def test_strict_path_tracks_unquantized_attention():
    lengths, hq, hkv, d = [300, 200], 4, 2, 64
    q, k, v, do, cu = _inputs(lengths, hq, hkv, d, seed=24)
    out = _strict(q, k, v, do, cu, hq, hkv)
    ref_o, _ = O.dense_attention(q, k, v, cu, hq, hkv)
    ref_g = O.dense_attention_grads(q, k, v, do, cu, hq, hkv)
    assert cosine(out["o"], ref_o) > 0.997
    for n in ("dq", "dk", "dv"):
        assert cosine(out[n], ref_g[n]) > 0.99, n


# ------------------------------------------------------------ mixed NVFP4 / FP8 route

def _mixed(q, k, v, do, cu, hq, hkv):
    return O.run_training_call(q, k, v, do, cu, hq, hkv, opts=O.Options(mixed=True))


def test_mixed_route_earlier_rows_are_bit_identical():
    """[KO] section 3.2 (NVFP4 scales stay inside one token) and [EN] section 4
    (the per-key V scale folded into P on diagonal tiles keeps masked keys at
    zero): in the mixed route a change to ANY later token of Q, K or V leaves O
    and LSE of every earlier row bit-identical -- not only rows of earlier
    32-token blocks, as in the default route.  The factor 2^12 lifts a shared
    exponent far enough that every other value of the group falls below the
    E4M3 normal range, so any shared scale on the path would show."""
    lengths, hq, hkv, d = [200, 70], 2, 1, 32
    q, k, v, do, cu = _inputs(lengths, hq, hkv, d, seed=40)
    base = _mixed(q, k, v, do, cu, hq, hkv)
    for t in (5, 40, 130, 199):
        for name in ("q", "k", "v"):
            x = {"q": q, "k": k, "v": v}
            y = x[name].copy()
            y[t] *= 2.0 ** 12
            x[name] = y
            pert = _mixed(x["q"], x["k"], x["v"], do, cu, hq, hkv)
            assert np.array_equal(pert["o"][:t], base["o"][:t]), (name, t)
            assert np.array_equal(pert["lse"][:, :t], base["lse"][:, :t]), (name, t)
            assert not np.array_equal(pert["o"][t:200], base["o"][t:200]), (name, t)   # positive control


def test_default_route_leaks_within_the_diagonal_block_mixed_does_not():
    """Negative control for the diagonal per-key V: the same V perturbation at
    token 40 changes rows 32..39 in the default route (shared block exponent)
    but not in the mixed route."""
    lengths, hq, hkv, d = [64], 1, 1, 16
    q, k, v, do, cu = _inputs(lengths, hq, hkv, d, seed=9)
    v2 = v.copy(); v2[40, 0, 0] *= 2.0 ** 12
    d0, d1 = _train(q, k, v, do, cu, hq, hkv), _train(q, k, v2, do, cu, hq, hkv)
    m0, m1 = _mixed(q, k, v, do, cu, hq, hkv), _mixed(q, k, v2, do, cu, hq, hkv)
    assert not np.array_equal(d0["o"][32:40], d1["o"][32:40])
    assert np.array_equal(m0["o"][:40], m1["o"][:40])


def test_mixed_route_scores_come_from_the_nvfp4_copies():
    """With Q and K on the E2M1 grid (every 16-group holding a 6, so the NVFP4
    scale is exactly 1 and the token-block E4M3 codes are exact too) the mixed
    and default routes see the same scores; with Q and K off that grid the
    NVFP4 rounding (coarser than E4M3) changes them."""
    rng = np.random.default_rng(41)
    T, hq, hkv, d = 96, 1, 1, 32
    grid = np.array([-6, -4, -3, -2, -1.5, -1, -0.5, 0, 0.5, 1, 1.5, 2, 3, 4, 6], float)
    mk = lambda: rng.choice(grid, size=(T, 1, d))
    q, k = mk(), mk()
    q[:, :, ::16] = 6.0; k[:, :, ::16] = 6.0
    v = O.bf16_round(rng.standard_normal((T, 1, d)))
    do = O.bf16_round(rng.standard_normal((T, 1, d)))
    cu = np.array([0, T])
    m = _mixed(q, k, v, do, cu, hq, hkv)
    assert np.array_equal(m["q_nvfp4_hat"], q) and np.array_equal(m["k_nvfp4_hat"], k)
    assert np.array_equal(m["q_hat"], q) and np.array_equal(m["k_hat"], k)
    # same scores: the routes differ only through the diagonal per-key V, so the
    # gradients of the first query tile's fully visible part agree closely
    dflt = _train(q, k, v, do, cu, hq, hkv)
    assert np.array_equal(m["lse"], dflt["lse"])
    qn = O.bf16_round(rng.standard_normal((T, 1, d)))
    m2 = _mixed(qn, k, v, do, cu, hq, hkv)
    d2 = _train(qn, k, v, do, cu, hq, hkv)
    assert not np.array_equal(m2["lse"], d2["lse"])


def test_mixed_route_tracks_unquantized_attention():
    """[EN] section 8 reports cosine 0.9920 (output) and 0.9906 (gradients) for the
    mixed route against an FP32 reference on 4x4096 causal inputs; small N(0,1)
    inputs land in the same range, below the MXFP8 route."""
    lengths, hq, hkv, d = [300, 212], 4, 2, 64
    q, k, v, do, cu = _inputs(lengths, hq, hkv, d, seed=42)
    out = _mixed(q, k, v, do, cu, hq, hkv)
    ref_o, _ = O.dense_attention(q, k, v, cu, hq, hkv)
    ref_g = O.dense_attention_grads(q, k, v, do, cu, hq, hkv)
    dflt = _train(q, k, v, do, cu, hq, hkv)
    co = cosine(out["o"], ref_o)
    assert 0.988 < co < 0.996 and co < cosine(dflt["o"], ref_o)
    for n in ("dq", "dk", "dv"):
        cg = cosine(out[n], ref_g[n])
        assert 0.986 < cg < 0.996 and cg < cosine(dflt[n], ref_g[n]), n


def test_mixed_and_strict_are_separate():
    q, k, v, do, cu = _inputs([40], 1, 1, 16, seed=43)
    with pytest.raises(ValueError):
        O.run_training_call(q, k, v, do, cu, 1, 1, opts=O.Options(mixed=True, strict=True))


# ------------------------------------------------------------ dS block quantizer (reading C-9)
#
# [EN] section 3 ("the analogous region is a 32 by 32 square") and section 5 (the
# 32 by 32 maxima of dS); [KO] section 3.3: dS is quantized with one round-up
# exponent per document-local 32x32 block (query block x key block).  The pins
# below fix the grouping, the exponent rule and the treatment of masked (zero)
# entries from values worked out by hand, and each plausible slip (one exponent
# per row, 32x128 blocks, one exponent per tile, the floor rule, an exponent off
# by one) is planted on the CPU and shown to fail them.

def _ds_hand_example():
    """A 64x64 dS tile (query rows 128..191, key columns 0..63 of a document)
    holding a few entries; every expected value below was worked out by hand
    from the E4M3 grid (3 mantissa bits, subnormal step 2**-9, max 448)."""
    x = np.zeros((64, 64))
    want = np.zeros((64, 64))
    # block (0, 0): amax 448 -> e = 0
    x[3, 5], want[3, 5] = 448.0, 448.0
    x[0, 1], want[0, 1] = 5 * 2.0 ** -9, 5 * 2.0 ** -9          # subnormal code 5, exact
    x[0, 7], want[0, 7] = 100.5, 104.0                          # grid step 8 in [64, 128)
    x[2, 2], want[2, 2] = -0.296875, -0.3125                    # 9.5 steps of 2**-5: tie -> even
    # block (0, 1): amax 900 = 1.7578 * 2**9 -> e = 2 (448 * 2 = 896 < 900)
    x[0, 40], want[0, 40] = 900.0, 896.0                        # 225 -> 224 (step 16)
    x[1, 33], want[1, 33] = 5 * 2.0 ** -9, 2.0 ** -7            # 1.25 subnormal steps -> 1, times 4
    x[5, 50], want[5, 50] = 5.25, 5.0                           # 1.3125: tie between 1.25 and 1.375
    x[7, 45], want[7, 45] = 6 * 2.0 ** -9, 2.0 ** -6            # 1.5 subnormal steps -> 2, times 4
    # block (1, 0): amax 1 -> e = -8 (448 / 256 = 1.75 >= 1 > 448 / 512)
    x[40, 2], want[40, 2] = 1.0, 1.0
    x[33, 0], want[33, 0] = 5 * 2.0 ** -17, 5 * 2.0 ** -17      # 5 * 2**-9 after scaling: exact
    x[63, 31], want[63, 31] = 25 * 2.0 ** -13, 0.0029296875     # 0.78125: tie -> 0.75, / 256
    # block (1, 1): no entry (masked keys) -> all zero
    return x, want


def _ds_blocks_pins(fn):
    """Every check the 32x32 dS block rule must pass, run against ``fn``."""
    x, want = _ds_hand_example()
    got = fn(x, 128, 0)
    assert np.array_equal(got, want), np.argwhere(got != want)[:4]
    rng = np.random.default_rng(50)
    for R, C, qoff, koff in ((128, 128, 0, 0), (97, 128, 256, 128), (128, 45, 384, 0), (3, 5, 128, 256)):
        ds = rng.standard_normal((R, C)) * np.exp2(rng.integers(-12, 12, (R, C)))
        ds[rng.random((R, C)) < 0.2] = 0.0                      # masked entries are exact zeros
        ds[: min(R, 32), : min(C, 32)] *= 2.0 ** 10              # one block far above the others
        out = fn(ds, qoff, koff)
        assert np.all(out[ds == 0] == 0)
        for r0 in range(0, R, 32):
            for c0 in range(0, C, 32):
                blk = ds[r0:r0 + 32, c0:c0 + 32]
                ob = out[r0:r0 + 32, c0:c0 + 32]
                # locality: the block's result depends on that block alone
                assert np.array_equal(ob, fn(blk, 0, 0))
                amax = np.abs(blk).max()
                if amax == 0:
                    continue
                # the exponent from an independent closed form (amax = f 2**k, f in [0.5, 1))
                f, k = np.frexp(amax)
                e = k - 9 + (f > 0.875)
                assert 224.0 < amax * 2.0 ** -e <= 448.0
                # every value sits on the E4M3 grid of that exponent, within half a step
                y = ob * 2.0 ** -e
                yb = np.abs(blk) * 2.0 ** -e
                step = np.exp2(np.maximum(np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -6))), -6) - 3)
                assert np.all(np.abs(y / step - np.round(y / step)) == 0)
                assert np.all(np.abs(np.abs(y) - yb) <= step / 2)
                # scaling the block by 2**j scales its result exactly (away from the subnormals)
                big = np.abs(blk) * 2.0 ** -e >= 2.0 ** -6
                assert np.array_equal(fn(blk * 8.0, 0, 0)[big], ob[big] * 8.0)


def test_ds_block_quantizer_pins():
    _ds_blocks_pins(O.flamia_oracle._quantize_ds_blocks)


def _mutant_per_row(dS, qoff, koff):
    e = O.roundup_exponent(np.abs(dS).max(axis=1))[:, None]
    return O.e4m3_round(dS * np.exp2(-e)) * np.exp2(e)


def _mutant_wide_blocks(dS, qoff, koff):          # 32 x 128 blocks
    out = np.zeros_like(dS)
    for r0 in range(0, dS.shape[0], 32):
        blk = dS[r0:r0 + 32]
        e = O.roundup_exponent(np.abs(blk).max())
        out[r0:r0 + 32] = O.e4m3_round(blk * 2.0 ** -e) * 2.0 ** e
    return out


def _mutant_per_tile(dS, qoff, koff):
    e = O.roundup_exponent(np.abs(dS).max())
    return O.e4m3_round(dS * 2.0 ** -e) * 2.0 ** e


def _mutant_rule(rule_shift, use_floor=False):
    def fn(dS, qoff, koff):
        out = np.zeros_like(dS)
        for r0 in range(0, dS.shape[0], 32):
            for c0 in range(0, dS.shape[1], 32):
                blk = dS[r0:r0 + 32, c0:c0 + 32]
                amax = np.abs(blk).max()
                e = (O.floor_exponent(amax) if use_floor else O.roundup_exponent(amax)) + rule_shift
                out[r0:r0 + 32, c0:c0 + 32] = O.e4m3_round(blk * 2.0 ** -e) * 2.0 ** e
        return out
    return fn


@pytest.mark.parametrize("mutant", [_mutant_per_row, _mutant_wide_blocks, _mutant_per_tile,
                                    _mutant_rule(1), _mutant_rule(-1), _mutant_rule(0, use_floor=True)],
                         ids=["per_row", "32x128", "per_tile", "exp_plus_1", "exp_minus_1", "floor_rule"])
def test_ds_block_pins_reject_planted_mistakes(mutant):
    with pytest.raises(AssertionError):
        _ds_blocks_pins(mutant)


def test_backward_uses_the_block_quantized_ds_for_dq_and_dk(monkeypatch):
    """Swapping the 32x32 rule for the per-row slip changes both dQ and dK of the
    training call: the block-quantized dS feeds both products (dK through its
    transpose, which the 32x32 square allows)."""
    lengths, hq, hkv, d = [150], 1, 1, 16
    q, k, v, do, cu = _inputs(lengths, hq, hkv, d, seed=51)
    do[:, :, :] *= np.exp2(np.random.default_rng(52).integers(-9, 9, (150, 1, 1)))   # spread the row scales
    base = _train(q, k, v, do, cu, hq, hkv)
    monkeypatch.setattr(O.flamia_oracle, "_quantize_ds_blocks", _mutant_per_row)
    pert = _train(q, k, v, do, cu, hq, hkv)
    assert not np.array_equal(base["dq"], pert["dq"])
    assert not np.array_equal(base["dk"], pert["dk"])
    assert np.array_equal(base["dv"], pert["dv"])          # dV does not use dS
