"""flamia_bwd_static_scratch: the backward for callers that cannot allocate
device memory (a plugin whose host hands it only its input and output
buffers, a loop that must avoid cudaMalloc's device-wide synchronisation).
Its scratch is the library's static device array, so the call needs no
workspace argument.  This file is collected last on purpose.

The test calls the new entry point through the C ABI twice in a row and
compares each result with the existing flamia_bwd (caller-provided workspace)
on the same inputs, within the parity tolerance of the other GPU tests."""
import ctypes

import numpy as np
import pytest

import flamia_workloads as W
from gpu_harness import cu_tensor, to_device_bf16
from metrics import norm_max_err

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module")
def F():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from microscaled_precision_causal_gb300 import build
    build.build()
    import microscaled_precision_causal_gb300 as F
    return F


def test_static_scratch_backward_matches_workspace_backward(F):
    import torch
    lengths, hq, hkv, d = [300, 77, 129, 1], 4, 2, 128
    T, N = sum(lengths), len(lengths)
    inp = W.make_inputs(W.custom([T], hq, hkv, d, seed=21))
    cu = cu_tensor(lengths)
    att = F.FlamiaAttention(T, N, hq, hkv, d)
    q, k, v, do = (to_device_bf16(inp[n]) for n in ("q", "k", "v", "do"))
    att.plan_build(cu)
    att.quantize(q, k, v, cu)
    att.forward(cu)
    att.backward(do, cu)
    torch.cuda.synchronize()
    ref = {n: t.float().cpu().numpy() for n, t in (("dq", att.dq), ("dk", att.dk), ("dv", att.dv))}
    qv, kv, vv = att.views()
    for call in range(2):
        dq = torch.full_like(att.dq, float("nan"))
        dk = torch.full_like(att.dk, float("nan"))
        dv = torch.full_like(att.dv, float("nan"))
        rc = F.lib().flamia_bwd_static_scratch(
            ctypes.byref(qv), ctypes.byref(kv), ctypes.byref(vv), att.out.data_ptr(), att.lse.data_ptr(),
            do.data_ptr(), cu.data_ptr(), N, T, hq, hkv, d, 1, 0.0, ctypes.byref(att.opts), att.plan.data_ptr(),
            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert rc == 0, F.lib().flamia_status_string(rc)
        torch.cuda.synchronize()
        assert att.device_status() == 0
        got = {"dq": dq, "dk": dk, "dv": dv}
        for n in ("dq", "dk", "dv"):
            g = got[n].float().cpu().numpy()
            assert np.all(np.isfinite(g)), (call, n)
            e = norm_max_err(g, ref[n])
            assert e <= TOL, f"call {call}: {n} differs from flamia_bwd by {e:.3e}"


def test_static_scratch_rejects_problems_beyond_its_size(F):
    """A problem whose workspace exceeds the static array is refused before any launch."""
    T, hq, hkv, d = 1 << 20, 32, 8, 128
    need = F.flamia_bwd_workspace_bytes(T, 1, hq, hkv, d)
    assert need > F.STATIC_SCRATCH_BYTES
    q = F.QTensor(256, 256, 256)
    rc = F.lib().flamia_bwd_static_scratch(ctypes.byref(q), ctypes.byref(q), ctypes.byref(q), 256, 256, 256, 256, 1,
                                           T, hq, hkv, d, 1, 0.0, None, 256, 256, 256, 256, None)
    assert rc == -4
