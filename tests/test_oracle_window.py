"""Pins for the oracle's noncausal and windowed calls (CPU only).

The pages time packed noncausal training calls beside the causal ones (FLAMIA
review section 8, Appendix H; Korean review section 4.8).  A call is described
by a (left, right) window: query i sees key j of its document iff
i - left <= j <= i + right, a negative bound meaning no limit; causal = (-1, 0),
noncausal = (-1, -1).  Each check ties the tiled oracle to a brute-force
definition or to a property of attention itself.
"""
import math

import numpy as np
import pytest

import oracle as O
from metrics import cosine, norm_max_err

WINDOWS = [(-1, -1), (70, 0), (40, 25), (-1, 10), (3, -1), (0, 0), (200, 130)]


def _inputs(lengths, hq, hkv, d, seed=0, bf16=True):
    rng = np.random.default_rng(seed)
    T = int(sum(lengths))
    mk = lambda h: rng.standard_normal((T, h, d))
    q, k, v, do = mk(hq), mk(hkv), mk(hkv), mk(hq)
    if bf16:
        q, k, v, do = (O.bf16_round(x) for x in (q, k, v, do))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(int)
    return q, k, v, do, cu


def _brute_visible(L, window):
    left, right = window
    i, j = np.meshgrid(np.arange(L), np.arange(L), indexing="ij")
    vis = np.ones((L, L), bool)
    if right >= 0:
        vis &= j <= i + right
    if left >= 0:
        vis &= j >= i - left
    return vis


@pytest.mark.parametrize("window", WINDOWS)
def test_visible_pairs_and_tile_ranges_brute_force(window):
    for L in (1, 5, 128, 129, 300, 517):
        vis = _brute_visible(L, window)
        assert O.visible_pairs([L], window) == int(vis.sum())
        lo, hi = O.visible_keys(np.arange(L), L, window)
        assert np.array_equal(lo, vis.argmax(1)) and np.array_equal(hi, L - 1 - vis[:, ::-1].argmax(1))
        nt = -(-L // 128)
        tiles = [[bool(vis[t * 128:(t + 1) * 128, u * 128:(u + 1) * 128].any()) for u in range(nt)] for t in range(nt)]
        for t in range(nt):
            assert [u for u in range(nt) if tiles[t][u]] == list(O.key_tiles(t, L, window))
        for u in range(nt):
            assert [t for t in range(nt) if tiles[t][u]] == list(O.query_tiles(u, L, window))
    assert O.visible_pairs([300, 40], (-1, -1)) == 300 ** 2 + 40 ** 2
    assert O.visible_pairs([300, 40]) == O.visible_pairs([300, 40], (-1, 0)) == 300 * 301 // 2 + 40 * 41 // 2


@pytest.mark.parametrize("window", WINDOWS)
def test_windowed_tiled_attention_equals_dense(window):
    lengths, hq, hkv, d = [300, 77, 129, 1], 2, 1, 16
    q, k, v, do, cu = _inputs(lengths, hq, hkv, d, seed=3)
    unq = O.Options(quantized=False, window=window)
    o1, l1 = O.attention_forward(q, k, v, cu, hq, hkv, opts=unq)
    o2, l2 = O.dense_attention(q, k, v, cu, hq, hkv, window=window)
    assert np.max(np.abs(o1 - o2)) <= 1e-12 * np.max(np.abs(o2))
    assert np.max(np.abs(l1 - l2)) <= 1e-12 * np.max(np.abs(l2))
    gt = O.attention_backward(q, k, v, o1, l1, do, cu, hq, hkv, opts=unq, diagnostics=True)
    gd = O.dense_attention_grads(q, k, v, do, cu, hq, hkv, window=window)
    for n in ("dq", "dk", "dv"):
        assert np.max(np.abs(gt[n] - gd[n])) <= 1e-11 * np.max(np.abs(gd[n])), n
    # the centred softmax gradient: every row of dS sums to zero
    rs, rm = gt["diag"]["rowsum_ds"], gt["diag"]["rowmax_ds"]
    assert np.max(np.abs(rs) / np.maximum(rm, 1e-300)) < 1e-12
    # the block size of the online recurrence does not matter
    for tile in (32, 64):
        o3, _ = O.attention_forward(q, k, v, cu, hq, hkv, opts=O.Options(quantized=False, window=window, tile=tile))
        assert np.max(np.abs(o3 - o2)) <= 1e-12 * np.max(np.abs(o2))


@pytest.mark.parametrize("window", [(-1, -1), (2, 1)])
def test_windowed_dense_gradients_match_finite_differences(window):
    lengths, hq, hkv, d = [7, 5], 2, 1, 4
    q, k, v, do, cu = _inputs(lengths, hq, hkv, d, seed=4, bf16=False)
    g = O.dense_attention_grads(q, k, v, do, cu, hq, hkv, window=window)
    loss = lambda q_, k_, v_: float((O.dense_attention(q_, k_, v_, cu, hq, hkv, window=window)[0] * do).sum())
    eps = 1e-6
    for name, x, gx in (("q", q, g["dq"]), ("k", k, g["dk"]), ("v", v, g["dv"])):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = {"q": q, "k": k, "v": v}
            args_p[name], args_m[name] = xp, xm
            num[idx] = (loss(**{a + "_": b for a, b in args_p.items()}) -
                        loss(**{a + "_": b for a, b in args_m.items()})) / (2 * eps)
        assert np.max(np.abs(num - gx)) <= 1e-6 * max(1.0, np.max(np.abs(gx))), name


def test_noncausal_attention_ignores_key_order():
    """Noncausal attention of a document is a function of its set of (key, value)
    pairs: permuting them leaves every output unchanged (unquantized)."""
    lengths, hq, hkv, d = [90, 60], 2, 2, 8
    q, k, v, do, cu = _inputs(lengths, hq, hkv, d, seed=5)
    unq = O.Options(quantized=False, window=(-1, -1))
    o1, l1 = O.attention_forward(q, k, v, cu, hq, hkv, opts=unq)
    perm = np.r_[np.random.default_rng(6).permutation(90), 90 + np.arange(60)]
    o2, l2 = O.attention_forward(q, k[perm], v[perm], cu, hq, hkv, opts=unq)
    assert np.max(np.abs(o1 - o2)) <= 1e-12 * np.max(np.abs(o1))
    assert np.max(np.abs(l1 - l2)) <= 1e-12 * np.max(np.abs(l1))
    # and a causal call does depend on the order
    oc1, _ = O.attention_forward(q, k, v, cu, hq, hkv, opts=O.Options(quantized=False))
    oc2, _ = O.attention_forward(q, k[perm], v[perm], cu, hq, hkv, opts=O.Options(quantized=False))
    assert np.max(np.abs(oc1 - oc2)) > 1e-3


def test_noncausal_quantized_call_tracks_unquantized_and_isolates_documents():
    lengths, hq, hkv, d = [300, 200], 4, 2, 64
    q, k, v, do, cu = _inputs(lengths, hq, hkv, d, seed=7)
    w = (-1, -1)
    out = O.run_training_call(q, k, v, do, cu, hq, hkv, opts=O.Options(window=w))
    ref_o, _ = O.dense_attention(q, k, v, cu, hq, hkv, window=w)
    ref_g = O.dense_attention_grads(q, k, v, do, cu, hq, hkv, window=w)
    assert cosine(out["o"], ref_o) > 0.997
    for n in ("dq", "dk", "dv"):
        assert cosine(out[n], ref_g[n]) > 0.99, n
        assert norm_max_err(out[n], ref_g[n]) < 0.15, n
    # another document's inputs change nothing of this one
    q2 = q.copy(); q2[:300] *= 8
    k2 = k.copy(); k2[:300] *= 0.25
    pert = O.run_training_call(q2, k2, v, do, cu, hq, hkv, opts=O.Options(window=w))
    s = slice(300, 500)
    for n in ("o", "dq", "dk", "dv"):
        assert np.array_equal(pert[n][s], out[n][s]), n
    # positive control: a later key of the same document changes an earlier row (not causal)
    k3 = k.copy(); k3[250] *= 4.0
    pert = O.run_training_call(q, k3, v, do, cu, hq, hkv, opts=O.Options(window=w))
    assert not np.array_equal(pert["o"][:32], out["o"][:32])


def test_windowed_work_list_costs():
    """Costs count the (query tile, key tile) pairs that hold a visible pair."""
    cu = [0, 1000, 1200, 1201, 5000]
    for window in ((-1, -1), (300, 0), (-1, 0)):
        items = O.work_list(cu, window=window)
        for it in items:
            s, t = cu[it["doc"]], cu[it["doc"] + 1]
            want = sum(len(O.key_tiles(tt, t - s, window)) for tt in range(it["tile0"], it["tile0"] + it["ntiles"]))
            assert it["cost"] == want
        costs = [it["cost"] for it in items]
        assert costs == sorted(costs, reverse=True)
        bw = O.bwd_key_tile_list(cu, window=window)
        assert [b["cost"] for b in bw] == sorted([b["cost"] for b in bw], reverse=True)
    nc = O.bwd_key_tile_list(cu, window=(-1, -1))
    assert all(b["cost"] == math.ceil((cu[b["doc"] + 1] - cu[b["doc"]]) / 128) for b in nc)


def test_strict_and_mixed_are_causal_only():
    q, k, v, do, cu = _inputs([40], 1, 1, 16, seed=8)
    for kw in (dict(strict=True), dict(mixed=True)):
        with pytest.raises(ValueError):
            O.run_training_call(q, k, v, do, cu, 1, 1, opts=O.Options(window=(-1, -1), **kw))
