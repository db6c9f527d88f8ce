"""The forward's two work-acquisition orders on the GPU (FLAMIA review section 6,
Algorithm 2): the static boustrophedon deal over persistent CTAs (step 06) and
dynamic acquisition through cluster launch control (steps 07 and 09).  A unit's
arithmetic does not depend on the CTA that runs it, so O and LSE are bitwise
identical under both; a second dynamic call on the same plan (the acquisition
counter is reset after every launch) gives the same bits again; and the dynamic
result matches the oracle."""
import numpy as np
import pytest

import flamia_workloads as W
from gpu_harness import cu_tensor, run_oracle, to_device_bf16
from metrics import norm_max_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from microscaled_precision_causal_gb300 import build
    build.build()


def _forward(w, inp, dynamic):
    import torch
    import microscaled_precision_causal_gb300 as F
    lengths = list(w.lengths)
    cu = cu_tensor(lengths)
    att = F.FlamiaAttention(w.total_tokens, len(lengths), w.hq, w.hkv, w.d, dynamic_schedule=dynamic)
    q, k, v = (to_device_bf16(inp[n]) for n in ("q", "k", "v"))
    att.plan_build(cu)
    att.quantize(q, k, v, cu)
    runs = []
    for _ in range(2 if dynamic else 1):
        att.forward(cu)
        torch.cuda.synchronize()
        assert att.device_status() == 0
        runs.append((att.out.view(torch.int16).cpu().numpy().copy(), att.lse.cpu().numpy().copy()))
    return runs


CASES = [
    ("packed_16k_h16_d128", None),
    ("skewed_8192_224x256_h16_d128", None),
    ("gqa_b4_s8192_hq32_hkv8_d128", None),
    ("ragged_d64", W.custom([700, 1, 129, 3000, 77], 4, 2, 64, seed=11, name="ragged_d64")),
    ("single_tile", W.custom([90], 2, 1, 128, seed=12, name="single_tile")),
]


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_dynamic_schedule_is_bitwise_the_static_one(name, w):
    w = w or W.WORKLOADS[name]
    inp = W.make_inputs(w)
    (o_s, l_s), = _forward(w, inp, False)
    (o_d, l_d), (o_d2, l_d2) = _forward(w, inp, True)
    assert np.array_equal(o_d, o_s)
    assert np.array_equal(l_d, l_s)
    assert np.array_equal(o_d2, o_d) and np.array_equal(l_d2, l_d)


def test_dynamic_schedule_matches_the_oracle():
    import torch
    w = W.custom([700, 1, 129, 3000, 77], 4, 2, 64, seed=11, name="ragged_d64")
    inp = W.make_inputs(w)
    (o_d, l_d), _ = _forward(w, inp, True)
    o = run_oracle(inp, list(w.lengths), w.hq, w.hkv, w.d, with_bwd=False)
    got = torch.from_numpy(o_d).view(torch.bfloat16).float().numpy().astype(np.float64)
    assert norm_max_err(got, o["o"]) <= 1e-2
    fin = np.isfinite(o["lse"])
    assert np.array_equal(fin, np.isfinite(l_d))
    assert np.max(np.abs(l_d[fin] - o["lse"][fin])) < 1e-3
