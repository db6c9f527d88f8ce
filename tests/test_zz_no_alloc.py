"""flamia_bwd_static_scratch: the backward for callers that cannot allocate
device memory (a plugin whose host hands it only its input and output
buffers, a loop that must avoid cudaMalloc's device-wide synchronisation).
Its scratch is the library's static device array, so the call needs no
workspace argument.  This file is collected last on purpose.

Each test first fills the shared array with another layout's data (a larger
call at the other head dimension), then calls the entry point through the C
ABI twice in a row and compares each result with the existing flamia_bwd
(caller-provided workspace) and with the oracle, within the parity tolerance
of the other GPU tests.  Between the two calls the device's free memory must
not change: the call allocates nothing."""
import ctypes

import numpy as np
import pytest

import flamia_workloads as W
import oracle as O
from gpu_harness import cu_tensor, run_oracle, to_device_bf16
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


class _Problem:
    """One layout: inputs on the device, the quantized views and the forward."""

    def __init__(self, F, lengths, hq, hkv, d, strict, seed):
        import torch
        self.lengths, self.hq, self.hkv, self.d = lengths, hq, hkv, d
        self.T, self.N = sum(lengths), len(lengths)
        self.inp = W.make_inputs(W.custom([self.T], hq, hkv, d, seed=seed))
        self.cu = cu_tensor(lengths)
        self.att = F.FlamiaAttention(self.T, self.N, hq, hkv, d, strict=strict)
        q, k, v = (to_device_bf16(self.inp[n]) for n in ("q", "k", "v"))
        self.do = to_device_bf16(self.inp["do"])
        self.att.plan_build(self.cu)
        self.att.quantize(q, k, v, self.cu)
        self.att.forward(self.cu)
        self.outs = [(torch.empty_like(self.att.dq), torch.empty_like(self.att.dk), torch.empty_like(self.att.dv))
                     for _ in range(2)]

    def call_static(self, F, i):
        import torch
        a = self.att
        dq, dk, dv = self.outs[i]
        for t in (dq, dk, dv):
            t.fill_(float("nan"))
        qv, kv, vv = a.views()
        return F.lib().flamia_bwd_static_scratch(
            ctypes.byref(qv), ctypes.byref(kv), ctypes.byref(vv), a.out.data_ptr(), a.lse.data_ptr(),
            self.do.data_ptr(), self.cu.data_ptr(), self.N, self.T, self.hq, self.hkv, self.d, 1, 0.0,
            ctypes.byref(a.opts), a.plan.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
            torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("strict", [False, True], ids=["default", "strict"])
def test_static_scratch_backward_matches_workspace_backward(F, d, strict):
    import torch
    # stale contents: a larger call with another layout (the other head dim, more heads)
    stale = _Problem(F, [700, 450, 97], 8, 2, 192 - d, strict, seed=20)
    assert stale.call_static(F, 0) == 0
    p = _Problem(F, [300, 77, 129, 1], 4, 2, d, strict, seed=21)
    p.att.backward(p.do, p.cu)                      # the existing entry point, caller-owned workspace
    torch.cuda.synchronize()
    ref = {n: t.float().cpu().numpy() for n, t in (("dq", p.att.dq), ("dk", p.att.dk), ("dv", p.att.dv))}
    orc = run_oracle(p.inp, p.lengths, p.hq, p.hkv, p.d, opts=O.Options(strict=strict))
    free = []
    for call in range(2):
        torch.cuda.synchronize()
        before = torch.cuda.mem_get_info()[0]
        rc = p.call_static(F, call)
        assert rc == 0, F.lib().flamia_status_string(rc)
        torch.cuda.synchronize()
        free.append((before, torch.cuda.mem_get_info()[0]))
        assert p.att.device_status() == 0
        for n, t in zip(("dq", "dk", "dv"), p.outs[call]):
            g = t.float().cpu().numpy()
            assert np.all(np.isfinite(g)), (call, n)
            e = norm_max_err(g, ref[n])
            assert e <= TOL, f"call {call}: {n} differs from flamia_bwd by {e:.3e}"
            e = norm_max_err(g, orc[n])
            assert e <= TOL, f"call {call}: {n} differs from the oracle by {e:.3e}"
    # the first call at a head dim may still load kernel code; the second one
    # must leave the device's free memory exactly as it found it
    assert free[1][0] == free[1][1], "device memory changed across a call"


def test_static_scratch_rejects_problems_beyond_its_size(F):
    """A problem whose workspace exceeds the static array is refused before any
    launch; a bad argument gets the same code as from flamia_bwd."""
    T, hq, hkv, d = 1 << 20, 32, 8, 128
    need = F.flamia_bwd_workspace_bytes(T, 1, hq, hkv, d)
    assert need > F.STATIC_SCRATCH_BYTES
    q = F.QTensor(256, 256, 256)
    call = lambda T_, hq_, hkv_, d_: F.lib().flamia_bwd_static_scratch(
        ctypes.byref(q), ctypes.byref(q), ctypes.byref(q), 256, 256, 256, 256, 1, T_, hq_, hkv_, d_, 1, 0.0, None,
        256, 256, 256, 256, None)
    assert call(T, hq, hkv, d) == -4                # FLAMIA_ERR_WORKSPACE
    assert call(T, hq, hkv, 96) == -2               # head_dim 96: FLAMIA_ERR_UNSUPPORTED, as flamia_bwd
    assert call(1024, 4, 3, 128) == -2              # hq % hkv != 0
    assert call(1024, 0, 1, 128) == -1              # FLAMIA_ERR_INVALID_ARG
