"""Pins for the oracle's codecs and exponent rules (CPU only).

Each check ties the oracle to something other than itself: a value the pages
print (tests/golden), a library decoder/encoder (torch / ml_dtypes float8), a
closed form, or an invariant that the pages state.
"""
import numpy as np
import pytest
import torch

import oracle as O
from golden_io import rows
from metrics import cosine, rel_l2

ALL_BYTES = np.arange(256, dtype=np.uint8)


def _torch_e4m3_decode():
    return torch.from_numpy(ALL_BYTES.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_matches_library_table():
    ours = O.e4m3_decode(ALL_BYTES)
    ref = _torch_e4m3_decode()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def test_e4m3_facts_from_pages():
    facts = {r[0]: float(r[1]) for r in rows("e4m3_facts.txt")}
    vals = O.e4m3_decode(ALL_BYTES)
    assert np.nanmax(vals) == facts["max_finite"]
    assert O.e4m3_encode(448.0) == 0x7E
    grid = np.unique(vals[~np.isnan(vals)])
    above_one = grid[grid > 1.0][0]
    assert above_one - 1.0 == facts["spacing_above_one"]
    assert grid[grid > 0][0] == facts["smallest_subnormal"]
    assert O.FP16_MAX == facts["fp16_max"]
    assert np.isinf(O.fp16_round(65520.0)) and O.fp16_round(65519.0) == 65504.0


def _all_finite_bf16_as_f64():
    b = np.arange(1 << 16, dtype=np.uint32)
    f = (b << 16).view(np.float32)
    return f[np.isfinite(f)].astype(np.float64)


@pytest.mark.parametrize("e", [-12, -6, -1, 0, 1, 3, 9])
def test_e4m3_round_matches_library_cast_in_range(e):
    """RNE against torch's float8_e4m3fn cast (non-saturating), in range only."""
    x = _all_finite_bf16_as_f64() * 2.0 ** -e
    x = x[np.abs(x) <= 448.0]
    ours = O.e4m3_round(x)
    ref = torch.from_numpy(x).to(torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)
    # codes (including the sign of zero) against the library's bytes
    ref_b = torch.from_numpy(x).to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(x), ref_b)


def test_e4m3_round_matches_ml_dtypes_if_present():
    ml = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(3)
    x = rng.standard_normal(200000) * np.exp2(rng.integers(-14, 9, 200000))
    x = x[np.abs(x) <= 448]
    ref = x.astype(np.float32).astype(ml.float8_e4m3fn).astype(np.float64)
    assert np.array_equal(O.e4m3_round(x), ref)


def test_e4m3_saturates():
    assert O.e4m3_round(449.0) == 448.0
    assert O.e4m3_round(1e9) == 448.0 and O.e4m3_round(-1e9) == -448.0
    assert O.e4m3_encode(-1e9) == 0xFE


def test_decode_encode_roundtrip_all_codes():
    v = O.e4m3_decode(ALL_BYTES)
    ok = ~np.isnan(v)
    assert np.array_equal(O.e4m3_encode(v[ok]), ALL_BYTES[ok])


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(300000) * np.exp2(rng.integers(-130, 120, 300000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.bf16_round(x.astype(np.float64)), ref)


def test_fp16_round_matches_numpy_and_torch():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(300000) * np.exp2(rng.integers(-30, 18, 300000))
    ours = O.fp16_round(x)
    with np.errstate(over="ignore"):
        assert np.array_equal(ours, x.astype(np.float16).astype(np.float64))
    # torch converts double -> half through float, so compare on fp32-exact inputs
    x32 = x.astype(np.float32).astype(np.float64)
    ref_t = torch.from_numpy(x32).to(torch.float32).to(torch.float16).to(torch.float64).numpy()
    assert np.array_equal(O.fp16_round(x32), ref_t)


def test_e2m1_ties_and_saturation():
    # ties go to the even code: 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4
    xs = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 100.0, -0.25, -5.0])
    want = np.array([0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0, -0.0, -4.0])
    got = O.e2m1_round(xs)
    assert np.array_equal(got, want) and np.array_equal(np.signbit(got), np.signbit(want))
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(O.e2m1_encode(O.e2m1_decode(codes))[codes != 8], codes[codes != 8])


# ---------------------------------------------------------------- exponent rules

def test_roundup_exponent_examples_and_closed_form():
    assert O.roundup_exponent(448.0) == 0
    assert O.roundup_exponent(449.0) == 1
    assert O.roundup_exponent(460.0) == 1
    assert O.roundup_exponent(900.0) == 2
    assert O.roundup_exponent(224.0) == -1
    assert O.roundup_exponent(0.0) == 0
    rng = np.random.default_rng(7)
    a = np.abs(rng.standard_normal(100000)) * np.exp2(rng.integers(-60, 60, 100000))
    a = np.concatenate([a, 448.0 * np.exp2(np.arange(-40, 40.0)), np.nextafter(448.0 * np.exp2(np.arange(-40, 40.0)), np.inf)])
    e = O.roundup_exponent(a)
    # independent closed form: a = f 2^k, f in [0.5,1): e = k - 9 + [f > 0.875]
    f, k = np.frexp(a)
    assert np.array_equal(e, k - 9 + (f > 0.875))
    # the defining inequality and minimality
    assert np.all(a <= 448.0 * np.exp2(e)) and np.all(a > 448.0 * np.exp2(e - 1))


def test_roundup_never_clamps_and_keeps_scaled_max_in_upper_binade():
    rng = np.random.default_rng(8)
    a = np.abs(rng.standard_normal(50000)) * np.exp2(rng.integers(-40, 40, 50000)) + 1e-30
    e = O.roundup_exponent(a)
    y = a * np.exp2(-e.astype(float))
    assert np.all(y <= 448.0) and np.all(y > 224.0)


def test_clamp_example_from_pages():
    for rule, group, value, exp, target, code, recon in rows("e4m3_clamp_example.txt"):
        amax = max(float(g) for g in group.split(","))
        fn = O.floor_exponent if rule == "floor" else O.roundup_exponent
        e = int(fn(amax))
        assert e == int(exp), (rule, group)
        t = float(value) * 2.0 ** -e
        assert t == float(target)
        assert int(O.e4m3_encode(t)) == int(code, 16)
        assert float(O.e4m3_decode(O.e4m3_encode(t))) * 2.0 ** e == float(recon)


def test_floor_rule_clamps_and_roundup_does_not():
    # a block whose max sits in (448, 512) * 2^k: the floor rule saturates it.
    x = np.array([[[460.0, 1.0]]])       # [T=1, H=1, d=2]
    cu = [0, 1]
    cf, sf = O.quantize_tokenblock(x, cu, rule="floor")
    cr, sr = O.quantize_tokenblock(x, cu, rule="roundup")
    assert O.dequantize_tokenblock(cf, sf)[0, 0, 0] == 448.0          # clipped
    recon = O.dequantize_tokenblock(cr, sr)[0, 0, 0]
    assert recon == 448.0 and cr[0, 0, 0] != 0x7E                        # rounded, not clipped


def test_doubling_the_scale_preserves_normal_codes():
    """[EN] section 4: with both codes normal and away from clipping, doubling
    the scale reconstructs the same value."""
    rng = np.random.default_rng(11)
    x = rng.uniform(1.0, 200.0, 20000) * np.where(rng.random(20000) < 0.5, -1, 1)
    for e in range(-4, 4):
        v1 = O.e4m3_round(x * 2.0 ** -e) * 2.0 ** e
        v2 = O.e4m3_round(x * 2.0 ** -(e + 1)) * 2.0 ** (e + 1)
        normal = (np.abs(x * 2.0 ** -(e + 1)) >= 2.0 ** -6) & (np.abs(x * 2.0 ** -e) <= 448)
        assert np.array_equal(v1[normal], v2[normal])


def test_doubling_the_scale_changes_the_subnormal_boundary():
    """[EN] section 4: a value held by the smallest subnormal code at scale s is
    halfway between zero and the smallest subnormal at scale 2s."""
    v = 2.0 ** -9
    assert O.e4m3_round(v) == v
    at_2s = O.e4m3_round(v / 2.0) * 2.0
    assert at_2s != v          # ties to even send it to zero


def test_p_budget_from_pages():
    for tau, beta_log2, w, boosted, stored, recon in rows("p_budget.txt"):
        beta = 2.0 ** int(beta_log2)
        assert beta * float(w) == float(boosted)
        assert O.e4m3_round(float(boosted)) == float(stored)
        assert O.e4m3_round(float(boosted)) / beta == float(recon)
        assert float(w) == 2.0 ** int(tau)


def test_cosine_example_from_pages():
    (rel, cos, zero_share), = rows("cosine_example.txt")
    full = np.array([1.0] + [0.001] * 100)
    dropped = np.array([1.0] + [0.0] * 100)
    assert abs(rel_l2(dropped, full) - float(rel)) < 1e-3
    assert abs(cosine(dropped, full) - float(cos)) < 1e-5
    assert abs(100 / 101 - float(zero_share)) < 1e-6


# ---------------------------------------------------------------- quantizer

def test_tokenblock_quantizer_structure():
    rng = np.random.default_rng(5)
    lengths = [45, 1, 70, 32, 33]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    T, H, d = int(cu[-1]) + 3, 3, 8          # three trailing tokens outside every document
    x = O.bf16_round(rng.standard_normal((T, H, d)) * 3.0)
    codes, sb = O.quantize_tokenblock(x, cu)
    for n in range(len(lengths)):
        for b0 in range(cu[n], cu[n + 1], 32):
            b1 = min(b0 + 32, cu[n + 1])
            for h in range(H):
                assert np.all(sb[b0:b1, h] == sb[b0, h])     # one exponent per block
                e = int(sb[b0, h]) - 127
                amax = np.abs(x[b0:b1, h]).max()
                assert amax <= 448 * 2.0 ** e < 2 * amax or amax == 0
    assert np.all(codes[int(cu[-1]):] == 0) and np.all(sb[int(cu[-1]):] == 127)
    # reconstruction error bounded by half an E4M3 step (relative 1/16) or the subnormal step
    xh = O.dequantize_tokenblock(codes, sb)
    scale = np.exp2(sb[:int(cu[-1])].astype(float) - 127)[:, :, None]
    err = np.abs(xh[:int(cu[-1])] - x[:int(cu[-1])])
    assert np.all(err <= np.maximum(np.abs(x[:int(cu[-1])]) / 16, scale * 2.0 ** -10) + 1e-300)


def test_quantizer_is_document_local():
    """Negative control of [EN] section 10: perturbing another document or moving a
    document's physical offset leaves its codes and scales bit-identical."""
    rng = np.random.default_rng(6)
    a = O.bf16_round(rng.standard_normal((50, 2, 16)))
    b = O.bf16_round(rng.standard_normal((40, 2, 16)))
    x1 = np.concatenate([a, b]); cu1 = [0, 50, 90]
    c1, s1 = O.quantize_tokenblock(x1, cu1)
    b2 = b * 64.0
    c2, s2 = O.quantize_tokenblock(np.concatenate([a, b2]), cu1)
    assert np.array_equal(c1[:50], c2[:50]) and np.array_equal(s1[:50], s2[:50])
    for shift in (1, 7, 31, 77):
        pre = O.bf16_round(rng.standard_normal((shift, 2, 16)))
        x3 = np.concatenate([pre, b]); cu3 = [0, shift, shift + 40]
        c3, s3 = O.quantize_tokenblock(x3, cu3)
        assert np.array_equal(c3[shift:], c1[50:]) and np.array_equal(s3[shift:], s1[50:])


def test_per_token_quantizer_is_token_local():
    rng = np.random.default_rng(9)
    x = O.bf16_round(rng.standard_normal((40, 2, 16)))
    c1, s1 = O.quantize_tokenblock(x, [0, 40], block=1)
    x2 = x.copy(); x2[20] *= 1000
    c2, s2 = O.quantize_tokenblock(x2, [0, 40], block=1)
    keep = np.arange(40) != 20
    assert np.array_equal(c1[keep], c2[keep]) and np.array_equal(s1[keep], s2[keep])


def test_nvfp4_quantizer_pins():
    rng = np.random.default_rng(10)
    x = O.bf16_round(rng.standard_normal((9, 2, 32)) * 5)
    codes, sc = O.quantize_nvfp4(x)
    s = O.e4m3_decode(sc)
    g = x.reshape(9, 2, 2, 16)
    amax = np.abs(g).max(-1)
    # the scale is the E4M3 value nearest amax/6; codes lie on the E2M1 grid
    assert np.array_equal(s, O.e4m3_round((amax.astype(np.float32) / np.float32(6)).astype(np.float64)))
    xh = O.dequantize_nvfp4(codes, sc)
    assert cosine(xh, x) > 0.97
    # the group maximum reconstructs within one E2M1 step of its scaled value
    assert np.all(np.abs(np.abs(xh.reshape(9, 2, 2, 16)).max(-1) - amax) <= 1.0 * s + 1e-12)


def test_nvfp4_hand_worked_groups():
    """Five 16-element groups whose scales and codes were worked out by hand from
    reading C-7 (s = E4M3(amax / 6), raised to 2**-9 for a non-zero group that
    would round to 0; codes = E2M1(x / s), ties to the even code, saturating):
    a scale tie that rounds down, one that rounds up, the 2**-9 floor, an
    all-zero group, and a scale that saturates at 448 (so the codes saturate at
    6 s).  Every input is exact in bf16."""
    groups = [
        # amax 6.375: 6.375 / 6 = 1.0625, tie between 1 and 1.125 -> 1 (even); 6.375 saturates to 6
        ([6.375, 1.3125, -2.625, 0.1875, 0.25, 0.75, 1.25, 2.5, 5.0, -0.75],
         1.0, 0x38, [6.0, 1.5, -3.0, 0.0, 0.0, 1.0, 1.0, 2.0, 4.0, -1.0], [7, 3, 13, 0, 0, 2, 2, 4, 6, 10]),
        # amax 7.125: 7.125 / 6 = 1.1875, tie between 1.125 and 1.25 -> 1.25 (even);
        # 7.125 / 1.25 = 5.7 -> 6; -3.125 / 1.25 = -2.5, tie -> -2; 0.625 / 1.25 = 0.5
        ([7.125, -3.125, 0.625], 1.25, 0x3A, [7.5, -2.5, 0.625], [7, 12, 1]),
        # amax 1.5 * 2**-10: amax / 6 = 2**-12 rounds to 0 in E4M3 -> floor 2**-9;
        # 0.75 steps -> 1 (tie to even), -0.25 steps -> -0 (tie to even)
        ([1.5 * 2.0 ** -10, -2.0 ** -11], 2.0 ** -9, 0x01, [2.0 ** -9, -0.0], [2, 8]),
        # all zero: scale code 0, codes 0
        ([], 0.0, 0x00, [], []),
        # amax 2944 = 1.4375 * 2**11: 2944 / 6 = 490.7 saturates to 448; 2944 / 448 = 6.57 -> 6
        ([2944.0, -1344.0], 448.0, 0x7E, [2688.0, -1344.0], [7, 13]),
    ]
    x = np.zeros((1, 1, 16 * len(groups)))
    for gi, (vals, *_rest) in enumerate(groups):
        x[0, 0, 16 * gi:16 * gi + len(vals)] = vals
    assert np.array_equal(O.bf16_round(x), x)
    codes, sc = O.quantize_nvfp4(x)
    xh = O.dequantize_nvfp4(codes, sc)
    for gi, (vals, s, s_code, recon, cds) in enumerate(groups):
        assert sc[0, 0, gi] == s_code and O.e4m3_decode(sc[0, 0, gi]) == s, gi
        n = len(vals)
        seg = slice(16 * gi, 16 * gi + n)
        assert np.array_equal(xh[0, 0, seg], recon), (gi, xh[0, 0, seg])
        assert np.array_equal(np.signbit(xh[0, 0, seg]), np.signbit(np.array(recon, float))), gi
        assert list(codes[0, 0, seg]) == cds, (gi, list(codes[0, 0, seg]))
        assert np.all(codes[0, 0, 16 * gi + n:16 * (gi + 1)] == 0), gi
