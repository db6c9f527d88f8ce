"""Run the CUDA path through the C ABI on seeded inputs and the oracle on the
same inputs (tests only)."""
import numpy as np

import flamia_workloads as W
import oracle as O


def bf16_values(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def to_device_bf16(bits, device="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)
    return t.view(torch.bfloat16)


def cu_tensor(lengths, device="cuda"):
    import torch
    return torch.tensor(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32), device=device)


def run_gpu(inputs, lengths, hq, hkv, d, total_tokens=None, with_bwd=True, scale=0.0, strict=False, mixed=False,
            window=(-1, 0), rotate=False):
    """inputs: dict of bf16 bit arrays (uint16) q, k, v[, do] of shape [T, H, d].  window:
    (left, right) visible keys, causal when right == 0 (the oracle's convention)."""
    import torch
    import microscaled_precision_causal_gb300 as F
    T = inputs["q"].shape[0] if total_tokens is None else total_tokens
    N = len(lengths)
    cu = cu_tensor(lengths)
    causal = window[1] == 0
    att = F.FlamiaAttention(T, N, hq, hkv, d, strict=strict, mixed=mixed, causal=causal, window=tuple(window),
                            rotate=rotate)
    q, k, v = (to_device_bf16(inputs[n]) for n in ("q", "k", "v"))
    att.plan_build(cu)
    att.quantize(q, k, v, cu)
    att.forward(cu, scale)
    out = {}
    if with_bwd:
        do = to_device_bf16(inputs["do"])
        att.backward(do, cu, scale)
        dc, ds = att.bwd_dout_codes()
        out.update(dq=att.dq, dk=att.dk, dv=att.dv, do_codes=dc, do_scales=ds)
    torch.cuda.synchronize()
    out.update(q_codes=att.q_codes, q_scales=att.q_scales, k_codes=att.k_codes, k_scales=att.k_scales,
               v_codes=att.v_codes, v_scales=att.v_scales, k_stats=att.k_stats, v_stats=att.v_stats,
               o=att.out, lse=att.lse, plan=att.plan)
    if mixed:
        out.update(q4_codes=att.q4_codes, q4_scales=att.q4_scales, k4_codes=att.k4_codes, k4_scales=att.k4_scales,
                   vt_codes=att.vt_codes, vt_scales=att.vt_scales)
    res = {}
    for key, val in out.items():
        if val.dtype == torch.bfloat16:
            res[key] = val.float().cpu().numpy().astype(np.float64)
        else:
            res[key] = val.cpu().numpy()
    res["status"] = att.device_status()
    return res


def run_oracle(inputs, lengths, hq, hkv, d, with_bwd=True, **sel):
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(int)
    vals = {n: bf16_values(inputs[n]) for n in inputs}
    return O.run_training_call(vals["q"], vals["k"], vals["v"], vals.get("do") if with_bwd else None, cu, hq, hkv,
                               **sel)
