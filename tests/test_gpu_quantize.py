"""GPU parity of the plan (work lists) and the token-block quantizer against
the oracle: bit-exact codes, scale bytes and item lists."""
import numpy as np
import pytest

import flamia_workloads as W
import oracle as O
from gpu_harness import bf16_values, cu_tensor, to_device_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from microscaled_precision_causal_gb300 import build
    build.build()
    import microscaled_precision_causal_gb300 as F
    return F


def _plan(F, lengths, T=None):
    import torch
    T = int(sum(lengths)) if T is None else T
    cu = cu_tensor(lengths)
    plan = torch.zeros(F.flamia_plan_bytes(T, len(lengths)), dtype=torch.uint8, device="cuda")
    F.flamia_plan_build(cu, len(lengths), T, plan)
    torch.cuda.synchronize()
    return cu, plan, plan.cpu().numpy().view(np.int32)


def _items(words, N, T):
    cap = T // 128 + N + 1
    pre = (16 + 3 * (N + 1) + 3) & ~3
    fwd = words[pre:pre + 4 * cap].reshape(cap, 4)
    bwd = words[pre + 4 * cap:pre + 8 * cap].reshape(cap, 4)
    return fwd[:words[6]], bwd[:words[7]]


@pytest.mark.parametrize("lengths,extra", [([300, 77, 129, 1], 0), ([256], 0), ([5000, 1, 0, 257, 128, 640], 37),
                                           ([8192] + [256] * 224, 0), (W.packed_lengths(16384, 128, 4096, 0), 0)])
def test_plan_matches_oracle_work_list(F, lengths, extra):
    T = int(sum(lengths)) + extra
    _, _, words = _plan(F, lengths, T)
    N = len(lengths)
    assert words[0] == 0 and words[1] == N and words[2] == T and words[3] == sum(lengths)
    assert words[4] == sum(-(-L // 32) for L in lengths)
    assert words[5] == sum(-(-L // 128) for L in lengths)
    fwd, bwd = _items(words, N, T)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    want = O.work_list(cu)
    assert [tuple(r) for r in fwd] == [(w["doc"], w["tile0"], w["ntiles"], w["cost"]) for w in want]
    wantb = O.bwd_key_tile_list(cu)
    assert [tuple(r[:3]) for r in bwd] == [(w["doc"], w["ktile"], w["cost"]) for w in wantb]


def test_plan_flags_malformed_cu_seqlens(F):
    import torch
    cu = torch.tensor([0, 50, 40, 100], dtype=torch.int32, device="cuda")
    plan = torch.zeros(F.flamia_plan_bytes(100, 3), dtype=torch.uint8, device="cuda")
    F.flamia_plan_build(cu, 3, 100, plan)
    assert F.flamia_get_device_status(plan) & F.DEV_BAD_CU_SEQLENS
    words = plan.cpu().numpy().view(np.int32)
    assert words[6] == 0 and words[7] == 0          # nothing scheduled


@pytest.mark.parametrize("lengths,H,d,extra,per_token", [
    ([300, 77, 129, 1], 3, 128, 0, False),
    ([300, 77, 129, 1], 2, 64, 21, False),
    ([31, 33, 1, 64, 200], 4, 128, 5, True),
    ([256], 2, 64, 0, True),
])
def test_quantizer_bit_exact(F, lengths, H, d, extra, per_token):
    import torch
    T = int(sum(lengths)) + extra
    w = W.custom([T], H, H, d, seed=11)
    bits = W.make_inputs(w, tensors=("q",))["q"]
    bits[:5] = W.f32_to_bf16_bits(np.float32([[[-0.0]]]) * np.ones((5, H, d), np.float32))   # signed zeros
    bits[6, 0, :4] = W.f32_to_bf16_bits(np.float32([1e-39, -3e-40, 2e-41, 448.0]))           # bf16 subnormals
    x = to_device_bf16(bits)
    cu, plan, _ = _plan(F, lengths, T)
    codes = torch.zeros(T, H, d, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(T, H, dtype=torch.uint8, device="cuda")
    stats = torch.zeros(T, H, 2, dtype=torch.float32, device="cuda")
    F.flamia_quantize_tokenblock(x, cu, len(lengths), plan, codes, scales, stats, per_token=per_token)
    torch.cuda.synchronize()
    xv = bf16_values(bits)
    oc, osb = O.quantize_tokenblock(xv, np.concatenate([[0], np.cumsum(lengths)]), block=1 if per_token else 32)
    gc, gs = codes.cpu().numpy(), scales.cpu().numpy()
    assert np.array_equal(gs, osb)
    mism = np.argwhere(gc != oc)
    assert mism.size == 0, f"{len(mism)} code mismatches, first {mism[:4].tolist()} gpu {gc[tuple(mism[0])]:#x} oracle {oc[tuple(mism[0])]:#x}"
    # stats: (||x^||_2, max |x^|) of the reconstructed rows
    xh = O.dequantize_tokenblock(oc, osb)
    st = stats.cpu().numpy()
    assert np.allclose(st[..., 0], np.sqrt((xh ** 2).sum(-1)), rtol=1e-5, atol=0)
    assert np.array_equal(st[..., 1], np.abs(xh).max(-1).astype(np.float32))


def test_quantizer_outlier_heavy_input(F):
    """Student-t(3) and x100 outliers: wide per-block exponent ranges, still bit-exact."""
    import torch
    lengths, H, d = [500, 300], 2, 128
    for dist in ("student_t3", "normal_outliers"):
        w = W.custom(lengths, H, H, d, dist=dist, seed=3)
        bits = W.make_inputs(w, tensors=("v",))["v"]
        cu, plan, _ = _plan(F, lengths)
        T = sum(lengths)
        codes = torch.zeros(T, H, d, dtype=torch.uint8, device="cuda")
        scales = torch.zeros(T, H, dtype=torch.uint8, device="cuda")
        F.flamia_quantize_tokenblock(to_device_bf16(bits), cu, 2, plan, codes, scales)
        oc, osb = O.quantize_tokenblock(bf16_values(bits), [0, 500, 800])
        assert np.array_equal(scales.cpu().numpy(), osb)
        assert np.array_equal(codes.cpu().numpy(), oc)


def _unpack_e2m1(packed):
    lo, hi = packed & 0x0F, packed >> 4
    return np.stack([lo, hi], axis=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)


@pytest.mark.parametrize("dist,d", [("normal", 128), ("normal_outliers", 128), ("student_t3", 64)])
def test_nvfp4_quantizer_bit_exact(F, dist, d):
    """NVFP4 score operands (reading C-7): E2M1 codes and E4M3 group scales equal
    the oracle's, bit for bit; element 2k sits in the low nibble of byte k."""
    import torch
    T, H = 777, 3
    w = W.custom([T], H, H, d, dist=dist, seed=5)
    bits = W.make_inputs(w, tensors=("q",))["q"]
    x = bf16_values(bits)
    x[3, 0, :16] = 0.0                                   # an all-zero group
    x[4, 1, 16:32] = x[4, 1, 16:32] * 2.0 ** -40         # scales below the E4M3 range: raised to 2^-9
    bits = W.f32_to_bf16_bits(x.astype(np.float32))
    codes = torch.zeros(T, H, d // 2, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(T, H, d // 16, dtype=torch.uint8, device="cuda")
    F.flamia_quantize_nvfp4(to_device_bf16(bits), codes, scales)
    torch.cuda.synchronize()
    oc, osc = O.quantize_nvfp4(bf16_values(bits))
    assert np.array_equal(scales.cpu().numpy(), osc)
    assert np.array_equal(_unpack_e2m1(codes.cpu().numpy()), oc)


@pytest.mark.parametrize("per_token", [False, True])
def test_fused_qkv_launch_equals_separate_calls(F, per_token):
    """flamia_quantize_qkv (Q, K and V in one launch) writes exactly what the three
    flamia_quantize_tokenblock calls write, including K / V row stats, on a GQA
    layout with tail tokens outside every document."""
    import torch
    lengths, hq, hkv, d = [300, 77, 129, 1], 4, 2, 128
    T = sum(lengths) + 9
    inp = W.make_inputs(W.custom([T], hq, hkv, d, dist="student_t3", seed=51))
    q, k, v = (to_device_bf16(inp[n]) for n in ("q", "k", "v"))
    cu, plan, _ = _plan(F, lengths, T)
    u8, f32 = torch.uint8, torch.float32
    mk = lambda H, *shape: torch.full((T, H) + shape, 0x5A, dtype=u8, device="cuda")
    sep = dict(qc=mk(hq, d), qs=mk(hq), kc=mk(hkv, d), ks=mk(hkv), vc=mk(hkv, d), vs=mk(hkv),
               kst=torch.full((T, hkv, 2), -1.0, dtype=f32, device="cuda"),
               vst=torch.full((T, hkv, 2), -1.0, dtype=f32, device="cuda"))
    fus = {n: t.clone() for n, t in sep.items()}
    N = len(lengths)
    F.flamia_quantize_tokenblock(q, cu, N, plan, sep["qc"], sep["qs"], None, per_token)
    F.flamia_quantize_tokenblock(k, cu, N, plan, sep["kc"], sep["ks"], sep["kst"], per_token)
    F.flamia_quantize_tokenblock(v, cu, N, plan, sep["vc"], sep["vs"], sep["vst"], per_token)
    F.flamia_quantize_qkv(q, k, v, cu, N, plan, fus["qc"], fus["qs"], fus["kc"], fus["ks"], fus["kst"], fus["vc"],
                          fus["vs"], fus["vst"], per_token)
    torch.cuda.synchronize()
    for n in sep:
        assert torch.equal(sep[n], fus[n]), n
    cuh = np.concatenate([[0], np.cumsum(lengths)])
    oc, osb = O.quantize_tokenblock(bf16_values(inp["k"]), cuh, 1 if per_token else 32)
    assert np.array_equal(fus["kc"].cpu().numpy(), oc) and np.array_equal(fus["ks"].cpu().numpy(), osb)
