"""GB300 (sm_103a) FLAMIA attention: thin Python binding of libflamia.

Argument marshalling only: every step of the path runs in the CUDA kernels of
``libflamia.so`` (built in-tree by ``build.py``).  PyTorch supplies device
memory and streams.  If the library is missing, every call raises -- there is
no CPU fallback.

The functions mirror the C ABI in ``include/flamia.h``:
``flamia_plan_bytes``, ``flamia_plan_build``, ``flamia_quantize_tokenblock``,
``flamia_fwd``, ``flamia_bwd_workspace_bytes``, ``flamia_bwd``,
``flamia_get_device_status``; ``FlamiaAttention`` strings them into the
training call (quantize Q/K/V, forward, backward).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libflamia.so")

FLAMIA_OK = 0
STATUS_NAMES = {0: "ok", -1: "invalid argument", -2: "unsupported", -3: "misaligned", -4: "workspace", -5: "cuda"}
DEV_BAD_CU_SEQLENS, DEV_TIMEOUT, DEV_CAPACITY = 1, 2, 4

EXPORTED = (
    "flamia_default_options", "flamia_plan_bytes", "flamia_plan_build", "flamia_quantize_tokenblock",
    "flamia_fwd", "flamia_bwd_workspace_bytes", "flamia_bwd", "flamia_get_device_status",
    "flamia_status_string", "flamia_bwd_static_scratch", "flamia_quantize_nvfp4", "flamia_plan_build_window",
    "flamia_quantize_hadamard", "flamia_quantize_qkv",
)
STATIC_SCRATCH_BYTES = 64 << 20


class FlamiaError(RuntimeError):
    pass


class Options(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "p_boost_log2", "bwd_p_boost_log2", "dq_headroom_log2", "strict_per_token", "strict_row_ds",
        "strict_causal_dq", "mixed_nvfp4", "deterministic")] + [("timing_events", ctypes.POINTER(ctypes.c_void_p)),
                                                                 ("mixed", ctypes.c_void_p),
                                                                 ("debug_p_ds", ctypes.c_void_p),
                                                                 ("window_left", ctypes.c_int),
                                                                 ("window_right", ctypes.c_int),
                                                                 ("rotate", ctypes.c_int),
                                                                 ("dynamic_schedule", ctypes.c_int)]


class QTensor(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("stats", ctypes.c_void_p)]


class MixedOperands(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("q_codes_e2m1", "q_scales_e4m3", "k_codes_e2m1", "k_scales_e4m3",
                                               "v_tok_codes", "v_tok_scales")]


_lib = None


def lib():
    """Load libflamia.so (raises FlamiaError if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise FlamiaError(f"{LIB_PATH} is missing: build it with microscaled_precision_causal_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    f32 = ctypes.c_float
    qp = ctypes.POINTER(QTensor)
    op = ctypes.POINTER(Options)
    sig = {
        "flamia_default_options": (None, [op]),
        "flamia_plan_bytes": (sz, [i64, i32]),
        "flamia_plan_build": (i32, [vp, i32, i64, vp, sz, vp]),
        "flamia_plan_build_window": (i32, [vp, i32, i64, i32, i32, i32, vp, sz, vp]),
        "flamia_quantize_tokenblock": (i32, [vp, i64, i32, i32, vp, i32, vp, i32, vp, vp, vp, vp]),
        "flamia_fwd": (i32, [qp, qp, qp, vp, i32, i64, i32, i32, i32, i32, f32, op, vp, vp, vp, vp]),
        "flamia_bwd_workspace_bytes": (sz, [i64, i32, i32, i32, i32]),
        "flamia_bwd": (i32, [qp, qp, qp, vp, vp, vp, vp, i32, i64, i32, i32, i32, i32, f32, op, vp, vp, vp, vp, vp,
                             sz, vp]),
        "flamia_bwd_static_scratch": (i32, [qp, qp, qp, vp, vp, vp, vp, i32, i64, i32, i32, i32, i32, f32, op, vp,
                                            vp, vp, vp, vp]),
        "flamia_get_device_status": (i32, [vp, ctypes.POINTER(ctypes.c_int), vp]),
        "flamia_status_string": (ctypes.c_char_p, [i32]),
        "flamia_quantize_nvfp4": (i32, [vp, i64, i32, i32, vp, vp, vp]),
        "flamia_quantize_hadamard": (i32, [vp, i64, i32, i32, vp, i32, vp, vp, vp, vp, vp]),
        "flamia_quantize_qkv": (i32, [vp, vp, vp, i64, i32, i32, i32, vp, i32, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                      vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _check(rc: int, what: str):
    if rc != FLAMIA_OK:
        raise FlamiaError(f"{what}: {lib().flamia_status_string(rc).decode()} ({rc})")


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def default_options() -> Options:
    o = Options()
    lib().flamia_default_options(ctypes.byref(o))
    return o


def qtensor(codes, scales, stats=None) -> QTensor:
    return QTensor(_ptr(codes), _ptr(scales), _ptr(stats))


# ---------------------------------------------------------------- C ABI mirrors

def flamia_plan_bytes(total_tokens: int, num_seqs: int) -> int:
    return int(lib().flamia_plan_bytes(total_tokens, num_seqs))


def flamia_plan_build(cu_seqlens, num_seqs: int, total_tokens: int, plan, stream=None):
    _check(lib().flamia_plan_build(_ptr(cu_seqlens), num_seqs, total_tokens, _ptr(plan), plan.numel() * plan.element_size(),
                                   _stream(stream)), "flamia_plan_build")


def flamia_plan_build_window(cu_seqlens, num_seqs: int, total_tokens: int, causal: int, window_left: int,
                             window_right: int, plan, stream=None):
    _check(lib().flamia_plan_build_window(_ptr(cu_seqlens), num_seqs, total_tokens, int(causal), window_left,
                                          window_right, _ptr(plan), plan.numel() * plan.element_size(),
                                          _stream(stream)), "flamia_plan_build_window")


def flamia_quantize_tokenblock(x, cu_seqlens, num_seqs: int, plan, codes, scales, stats=None, per_token: bool = False,
                               stream=None):
    T, H, d = x.shape
    _check(lib().flamia_quantize_tokenblock(_ptr(x), T, H, d, _ptr(cu_seqlens), num_seqs, _ptr(plan), int(per_token),
                                            _ptr(codes), _ptr(scales), _ptr(stats), _stream(stream)),
           "flamia_quantize_tokenblock")


def flamia_quantize_qkv(q, k, v, cu_seqlens, num_seqs: int, plan, q_codes, q_scales, k_codes, k_scales, k_stats,
                        v_codes, v_scales, v_stats, per_token: bool = False, stream=None):
    T, hq, d = q.shape
    hkv = k.shape[1]
    _check(lib().flamia_quantize_qkv(_ptr(q), _ptr(k), _ptr(v), T, hq, hkv, d, _ptr(cu_seqlens), num_seqs, _ptr(plan),
                                     int(per_token), _ptr(q_codes), _ptr(q_scales), _ptr(k_codes), _ptr(k_scales),
                                     _ptr(k_stats), _ptr(v_codes), _ptr(v_scales), _ptr(v_stats), _stream(stream)),
           "flamia_quantize_qkv")


def flamia_quantize_hadamard(x, cu_seqlens, num_seqs: int, plan, codes, scales, stats=None, stream=None):
    T, H, d = x.shape
    _check(lib().flamia_quantize_hadamard(_ptr(x), T, H, d, _ptr(cu_seqlens), num_seqs, _ptr(plan), _ptr(codes),
                                          _ptr(scales), _ptr(stats), _stream(stream)), "flamia_quantize_hadamard")


def flamia_quantize_nvfp4(x, codes, scales, stream=None):
    T, H, d = x.shape
    _check(lib().flamia_quantize_nvfp4(_ptr(x), T, H, d, _ptr(codes), _ptr(scales), _stream(stream)),
           "flamia_quantize_nvfp4")


def flamia_fwd(q: QTensor, k: QTensor, v: QTensor, cu_seqlens, num_seqs: int, total_tokens: int, hq: int, hkv: int,
               head_dim: int, plan, out, lse, softmax_scale: float = 0.0, opts: Optional[Options] = None,
               causal: int = 1, stream=None):
    _check(lib().flamia_fwd(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), _ptr(cu_seqlens), num_seqs, total_tokens,
                            hq, hkv, head_dim, causal, softmax_scale, ctypes.byref(opts) if opts else None, _ptr(plan),
                            _ptr(out), _ptr(lse), _stream(stream)), "flamia_fwd")


def flamia_bwd_workspace_bytes(total_tokens: int, num_seqs: int, hq: int, hkv: int, head_dim: int) -> int:
    return int(lib().flamia_bwd_workspace_bytes(total_tokens, num_seqs, hq, hkv, head_dim))


def flamia_bwd(q: QTensor, k: QTensor, v: QTensor, out, lse, dout, cu_seqlens, num_seqs: int, total_tokens: int,
               hq: int, hkv: int, head_dim: int, plan, dq, dk, dv, workspace, softmax_scale: float = 0.0,
               opts: Optional[Options] = None, causal: int = 1, stream=None):
    _check(lib().flamia_bwd(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), _ptr(out), _ptr(lse), _ptr(dout),
                            _ptr(cu_seqlens), num_seqs, total_tokens, hq, hkv, head_dim, causal, softmax_scale,
                            ctypes.byref(opts) if opts else None, _ptr(plan), _ptr(dq), _ptr(dk), _ptr(dv),
                            _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
           "flamia_bwd")


def flamia_bwd_static_scratch(q: QTensor, k: QTensor, v: QTensor, out, lse, dout, cu_seqlens, num_seqs: int,
                              total_tokens: int, hq: int, hkv: int, head_dim: int, plan, dq, dk, dv,
                              softmax_scale: float = 0.0, opts: Optional[Options] = None, causal: int = 1,
                              stream=None):
    """flamia_bwd without a workspace argument, for callers that cannot allocate
    device memory: the scratch is the library's static device array
    (STATIC_SCRATCH_BYTES per GPU).  The first call on a device must come before
    any stream capture; calls that overlap on the GPU race on the shared array."""
    _check(lib().flamia_bwd_static_scratch(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), _ptr(out), _ptr(lse),
                                           _ptr(dout), _ptr(cu_seqlens), num_seqs, total_tokens, hq, hkv, head_dim,
                                           causal, softmax_scale, ctypes.byref(opts) if opts else None, _ptr(plan),
                                           _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream)),
           "flamia_bwd_static_scratch")


def flamia_get_device_status(plan, stream=None) -> int:
    st = ctypes.c_int(0)
    _check(lib().flamia_get_device_status(_ptr(plan), ctypes.byref(st), _stream(stream)), "flamia_get_device_status")
    return st.value


# ---------------------------------------------------------------- training call

class FlamiaAttention:
    """Buffers and calls for one packed attention layout.

    All tensors live on one CUDA device; the object owns the plan, the
    quantized Q/K/V views and the backward workspace (allocated once through
    torch, reused across calls: nothing is allocated per call).  causal=False
    gives attention over the whole document; window = (left, right) limits the
    visible keys to i - left <= j <= i + right (-1: no limit; causal calls use
    right = 0).  dynamic_schedule=True makes the causal MXFP8 forward acquire
    its work through cluster launch control instead of the static order (same
    results)."""

    def __init__(self, total_tokens: int, num_seqs: int, hq: int, hkv: int, head_dim: int, device="cuda",
                 strict: bool = False, mixed: bool = False, causal: bool = True, window=(-1, -1),
                 rotate: bool = False, dynamic_schedule: bool = False):
        import torch
        self.T, self.N, self.hq, self.hkv, self.d = total_tokens, num_seqs, hq, hkv, head_dim
        self.causal = 1 if causal else 0
        self.window = (int(window[0]), int(window[1]))
        self.device = torch.device(device)
        dev = self.device
        u8 = torch.uint8
        self.plan = torch.empty(flamia_plan_bytes(total_tokens, num_seqs), dtype=u8, device=dev)
        self.q_codes = torch.empty(total_tokens, hq, head_dim, dtype=u8, device=dev)
        self.q_scales = torch.empty(total_tokens, hq, dtype=u8, device=dev)
        self.k_codes = torch.empty(total_tokens, hkv, head_dim, dtype=u8, device=dev)
        self.k_scales = torch.empty(total_tokens, hkv, dtype=u8, device=dev)
        self.k_stats = torch.empty(total_tokens, hkv, 2, dtype=torch.float32, device=dev)
        self.v_codes = torch.empty(total_tokens, hkv, head_dim, dtype=u8, device=dev)
        self.v_scales = torch.empty(total_tokens, hkv, dtype=u8, device=dev)
        self.v_stats = torch.empty(total_tokens, hkv, 2, dtype=torch.float32, device=dev)
        self.out = torch.empty(total_tokens, hq, head_dim, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(hq, total_tokens, dtype=torch.float32, device=dev)
        self.dq = torch.empty(total_tokens, hq, head_dim, dtype=torch.bfloat16, device=dev)
        self.dk = torch.empty(total_tokens, hkv, head_dim, dtype=torch.bfloat16, device=dev)
        self.dv = torch.empty(total_tokens, hkv, head_dim, dtype=torch.bfloat16, device=dev)
        ws = flamia_bwd_workspace_bytes(total_tokens, num_seqs, hq, hkv, head_dim)
        self.workspace = torch.empty(ws, dtype=u8, device=dev)
        self.opts = default_options()
        self.opts.window_left, self.opts.window_right = self.window
        self.rotate = bool(rotate)      # Q and K rotated by the Hadamard map before quantization
        self.opts.rotate = int(self.rotate)
        self.opts.dynamic_schedule = int(bool(dynamic_schedule))
        self.strict = bool(strict)
        if self.strict:   # per-token operand scales, per-query-row dS exponents, causal dQ boost, deterministic dQ
            for f in ("strict_per_token", "strict_row_ds", "strict_causal_dq", "deterministic"):
                setattr(self.opts, f, 1)
        self.mixed = bool(mixed)
        if self.mixed:    # NVFP4 score operands, per-token V copy for the diagonal key tiles
            T = total_tokens
            self.q4_codes = torch.empty(T, hq, head_dim // 2, dtype=u8, device=dev)
            self.q4_scales = torch.empty(T, hq, head_dim // 16, dtype=u8, device=dev)
            self.k4_codes = torch.empty(T, hkv, head_dim // 2, dtype=u8, device=dev)
            self.k4_scales = torch.empty(T, hkv, head_dim // 16, dtype=u8, device=dev)
            self.vt_codes = torch.empty(T, hkv, head_dim, dtype=u8, device=dev)
            self.vt_scales = torch.empty(T, hkv, dtype=u8, device=dev)
            self._mixed_ops = MixedOperands(_ptr(self.q4_codes), _ptr(self.q4_scales), _ptr(self.k4_codes),
                                            _ptr(self.k4_scales), _ptr(self.vt_codes), _ptr(self.vt_scales))
            self.opts.mixed_nvfp4 = 1
            self.opts.mixed = ctypes.cast(ctypes.pointer(self._mixed_ops), ctypes.c_void_p)

    def views(self):
        return (qtensor(self.q_codes, self.q_scales), qtensor(self.k_codes, self.k_scales, self.k_stats),
                qtensor(self.v_codes, self.v_scales, self.v_stats))

    def plan_build(self, cu_seqlens, stream=None):
        if self.causal and self.window[0] < 0:
            flamia_plan_build(cu_seqlens, self.N, self.T, self.plan, stream)
        else:
            flamia_plan_build_window(cu_seqlens, self.N, self.T, self.causal, self.window[0], self.window[1], self.plan,
                                     stream)

    def quantize(self, q, k, v, cu_seqlens, stream=None):
        pt = self.strict
        if self.rotate:
            flamia_quantize_hadamard(q, cu_seqlens, self.N, self.plan, self.q_codes, self.q_scales, None, stream)
            flamia_quantize_hadamard(k, cu_seqlens, self.N, self.plan, self.k_codes, self.k_scales, self.k_stats,
                                     stream)
            flamia_quantize_tokenblock(v, cu_seqlens, self.N, self.plan, self.v_codes, self.v_scales, self.v_stats, pt,
                                       stream)
        else:             # Q, K and V in one launch
            flamia_quantize_qkv(q, k, v, cu_seqlens, self.N, self.plan, self.q_codes, self.q_scales, self.k_codes,
                                self.k_scales, self.k_stats, self.v_codes, self.v_scales, self.v_stats, pt, stream)
        if self.mixed:
            flamia_quantize_nvfp4(q, self.q4_codes, self.q4_scales, stream)
            flamia_quantize_nvfp4(k, self.k4_codes, self.k4_scales, stream)
            flamia_quantize_tokenblock(v, cu_seqlens, self.N, self.plan, self.vt_codes, self.vt_scales, None, True,
                                       stream)

    def forward(self, cu_seqlens, softmax_scale: float = 0.0, stream=None):
        q, k, v = self.views()
        flamia_fwd(q, k, v, cu_seqlens, self.N, self.T, self.hq, self.hkv, self.d, self.plan, self.out, self.lse,
                   softmax_scale, self.opts, causal=self.causal, stream=stream)
        return self.out, self.lse

    def backward(self, dout, cu_seqlens, softmax_scale: float = 0.0, stream=None):
        q, k, v = self.views()
        flamia_bwd(q, k, v, self.out, self.lse, dout, cu_seqlens, self.N, self.T, self.hq, self.hkv, self.d, self.plan,
                   self.dq, self.dk, self.dv, self.workspace, softmax_scale, self.opts, causal=self.causal,
                   stream=stream)
        return self.dq, self.dk, self.dv

    def training_call(self, q, k, v, dout, cu_seqlens, softmax_scale: float = 0.0, stream=None, build_plan=True):
        """Plan (optional), quantize Q/K/V, forward and backward: one pass of the hot path."""
        if build_plan:
            self.plan_build(cu_seqlens, stream)
        self.quantize(q, k, v, cu_seqlens, stream)
        self.forward(cu_seqlens, softmax_scale, stream)
        return self.backward(dout, cu_seqlens, softmax_scale, stream)

    def device_status(self, stream=None) -> int:
        return flamia_get_device_status(self.plan, stream)

    def bwd_dvec(self):
        """View into the backward workspace: D = rowsum(dO^ o O), float [hq, T], of the last backward call."""
        import torch
        T, H, d = self.T, self.hq, self.d
        rnd = lambda x: (x + 255) // 256 * 256
        off = rnd(rnd(rnd(T * H * d) + T * H) + T * H * 8)
        return self.workspace[off:off + T * H * 4].view(torch.float32).view(H, T)

    def bwd_dout_codes(self):
        """Views into the backward workspace: (dO codes, dO scale bytes) of the last backward call."""
        import torch
        T, H, d = self.T, self.hq, self.d
        rnd = lambda x: (x + 255) // 256 * 256
        n_codes = T * H * d
        codes = self.workspace[:n_codes].view(T, H, d)
        off = rnd(n_codes)
        scales = self.workspace[off:off + T * H].view(T, H)
        return codes, scales
