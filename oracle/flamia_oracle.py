"""fp64 CPU oracle for FLAMIA: causal flash attention with microscaled FP8 operands.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  It
shares no code with the CUDA library (no kernels, headers, tables or helpers);
the only module both sides use is the seeded input generator
``flamia_workloads``, which holds none of the method's arithmetic.

Sources (web pages about the paper "FLAMIA: FLAsh MIcroscaling Attention for
Fast and Causally Safe Training on Blackwell", arXiv 2611.03344):
  [EN] "FLAMIA technical review" (Zhongzhu Zhou, 2026-11-08), sections 1-11,
       Algorithm 1 ("Microscaled forward and recomputed backward") and
       Algorithm 2 ("Document-local work list and launch").
  [KO] Korean review of the same paper (jaehun.me), sections 1-5.
  [FA] "Model development: efficient execution" (blog post on FlashAttention
       and low-precision formats), sections "Attention without the score
       matrix" and "Lower precision".

Everything is float64 numpy except where the method fixes a narrower format
(E4M3 / E2M1 / UE8M0 codes, bf16 outputs, fp16 dQ partials); those are
emulated exactly.  Where the pages are silent or garbled, the reading taken
is named in the docstring (C-1 ... C-19, listed with reasons in the design
notes).

Parity status: the codecs, exponent rules, cost model, work list, the
unquantized attention path and the prefix-isolation properties are pinned by
tests against the pages and mathematics.  The quantized attention as a whole
has no external anchor beyond its parts (the pages print no quantized output
values) -- its end-to-end values are "parity unpinned" beyond those parts.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Iterable, List, Optional, Sequence, Tuple

import numpy as np

__all__ = [
    "E4M3_MAX", "FP16_MAX", "e4m3_decode", "e4m3_round", "e4m3_encode", "e2m1_round", "e2m1_encode",
    "e2m1_decode", "bf16_round", "fp16_round", "ue8m0_decode",
    "roundup_exponent", "floor_exponent", "quantize_tokenblock", "dequantize_tokenblock", "hadamard_rotate", "hadamard_norm_log2",
    "quantize_nvfp4", "dequantize_nvfp4",
    "Options", "attention_forward", "attention_backward", "run_training_call",
    "dense_attention", "dense_attention_grads", "visible_pairs", "work_list",
    "bwd_key_tile_list", "visible_keys", "key_tiles", "query_tiles", "dq_boost", "causal_dq_boost", "doc_ranges",
]

E4M3_MAX = 448.0          # largest finite E4M3 magnitude ([FA] "Lower precision", format table)
E4M3_EMAX = 8             # binade of the largest code: 448 = 1.75 * 2**8
FP16_MAX = 65504.0        # [FA] "Lower precision", format table
BF16_MAX = float(np.ldexp(2.0 - 2.0 ** -7, 127))


# --------------------------------------------------------------------------
# Codecs.  [EN] section 2 "Codes, scales, and hardware layout"; [FA] "Lower
# precision".  Reading C-1: OCP E4M3 "fn" (bias 7, max 448, NaN = S.1111.111,
# no infinities, subnormals m * 2**-9), round to nearest with ties to even,
# saturating to +-448.
# --------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """E4M3 byte -> value (fp64)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    ef = (c >> 3) & 0xF
    mf = c & 0x7
    mag = np.where(ef == 0, mf * 2.0 ** -9, (1.0 + mf / 8.0) * np.ldexp(1.0, ef - 7))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


def e4m3_round(x) -> np.ndarray:
    """Nearest E4M3 value to x (ties to even), saturated to +-448; sign of zero kept."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, k = np.frexp(a)                      # a = f * 2**k with f in [0.5, 1)
    binade = np.maximum(k - 1, -6)          # below 2**-6 the grid is the subnormal one
    step = np.ldexp(1.0, binade - 3)        # 3 mantissa bits
    with np.errstate(invalid="ignore"):
        r = np.round(a / step) * step       # numpy rounds halves to even
    r = np.where(np.isnan(a), np.nan, np.minimum(r, E4M3_MAX))
    return np.copysign(r, x)


def e4m3_encode(x) -> np.ndarray:
    """Value -> E4M3 byte after :func:`e4m3_round`."""
    v = e4m3_round(x)
    a = np.abs(v)
    neg = np.signbit(v)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    _, k = np.frexp(a)
    binade = k - 1
    normal = a >= 2.0 ** -6
    ef = np.where(normal, binade + 7, 0)
    mant = np.where(normal, (a / np.ldexp(1.0, np.where(normal, binade, 0)) - 1.0) * 8.0,
                    a / 2.0 ** -9)
    code = (ef.astype(np.int64) << 3) | np.rint(mant).astype(np.int64)
    code = np.where(nan, 0x7F, code)
    code = code | np.where(neg, 0x80, 0)
    return code.astype(np.uint8)


def ue8m0_decode(b) -> np.ndarray:
    """UE8M0 scale byte -> 2**(b-127) (0xFF is NaN)."""
    b = np.asarray(b, dtype=np.int64)
    return np.where(b == 0xFF, np.nan, np.ldexp(1.0, b - 127))


_E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_round(x) -> np.ndarray:
    """Nearest E2M1 value (ties to the even code), saturated to +-6 ([EN] section 2:
    NVFP4 = E2M1 codes with an E4M3 scale per 16 elements)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    step = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    r = np.minimum(np.round(a / step) * step, 6.0)
    return np.copysign(r, x)


def e2m1_encode(x) -> np.ndarray:
    """Value -> 4-bit E2M1 code (bit 3 = sign), one code per uint8."""
    v = e2m1_round(x)
    idx = np.searchsorted(_E2M1_VALUES, np.abs(v))
    return (idx | np.where(np.signbit(v), 8, 0)).astype(np.uint8)


def e2m1_decode(c) -> np.ndarray:
    c = np.asarray(c, dtype=np.int64)
    return np.where(c & 8, -1.0, 1.0) * _E2M1_VALUES[c & 7]


def _round_to_bits(x, mant_bits: int, min_binade: int, max_finite: float) -> np.ndarray:
    """Round fp64 to a binary float with ``mant_bits`` stored mantissa bits (nearest even)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, k = np.frexp(a)
    binade = np.maximum(k - 1, min_binade)
    step = np.ldexp(1.0, binade - mant_bits)
    with np.errstate(invalid="ignore", over="ignore"):
        r = np.round(a / step) * step
    r = np.where(r > max_finite, np.inf, r)
    r = np.where(np.isnan(a), np.nan, r)
    return np.copysign(r, x)


def bf16_round(x) -> np.ndarray:
    """fp64 -> nearest bf16 value (ties to even); overflow -> inf."""
    return _round_to_bits(x, 7, -126, BF16_MAX)


def fp16_round(x) -> np.ndarray:
    """fp64 -> nearest IEEE half value (ties to even); overflow -> inf."""
    return _round_to_bits(x, 10, -14, FP16_MAX)


# --------------------------------------------------------------------------
# Exponent rules.  [EN] section 4 "Why doubling the scale often preserves
# E4M3 values" (clipping as the second failure; the conservative scale) and
# [KO] section 3.2 (rounding the exponent up keeps the scaled maximum <= 448).
# --------------------------------------------------------------------------

def roundup_exponent(amax) -> np.ndarray:
    """Reading C-2: the smallest integer e with amax <= 448 * 2**e.

    A zero block takes e = 0 (the pages allow "a conventional finite scale");
    e is clamped to the UE8M0 range [-127, 127]."""
    amax = np.asarray(amax, dtype=np.float64)
    pos = amax > 0
    safe = np.where(pos, amax, 448.0)
    # log2 of each factor separately: amax / 448 can underflow for tiny (subnormal) amax
    e = np.clip(np.ceil(np.log2(safe) - np.log2(E4M3_MAX)), -128, 128).astype(np.int64)
    # log2 is not exact: settle the inequality with exact power-of-two products.
    for _ in range(2):
        e = np.where(safe > np.ldexp(E4M3_MAX, e), e + 1, e)
        e = np.where(safe <= np.ldexp(E4M3_MAX, e - 1), e - 1, e)
    e = np.where(pos, e, 0)
    return np.clip(e, -127, 127)


def floor_exponent(amax) -> np.ndarray:
    """Negative control only: the floor rule e = floor(log2 amax) - emax with
    emax = 8 for E4M3 ([KO] section 2; [EN] section 4 "A floor rule based only
    on the largest code exponent").  It lets amax * 2**-e exceed 448."""
    amax = np.asarray(amax, dtype=np.float64)
    _, k = np.frexp(np.where(amax > 0, amax, 1.0))
    e = (k - 1) - E4M3_EMAX
    return np.clip(np.where(amax > 0, e, 0), -127, 127)


# --------------------------------------------------------------------------
# Packed documents.  [EN] section 6 "Preserve the logical row before
# optimizing the physical tile": token blocks are local to each document; the
# scale metadata is dense (one entry per token).
# --------------------------------------------------------------------------

def doc_ranges(cu) -> List[Tuple[int, int]]:
    cu = [int(c) for c in cu]
    return [(cu[n], cu[n + 1]) for n in range(len(cu) - 1)]


def _doc_blocks(cu, block: int):
    for s, t in doc_ranges(cu):
        for b0 in range(s, t, block):
            yield b0, min(b0 + block, t)


def quantize_tokenblock(x, cu, block: int = 32, rule: str = "roundup"):
    """Token-block MXFP8 quantizer ([EN] section 3 "Why one shared exponent can
    serve two reductions"; [KO] section 3.1; Algorithm 1 step 03).

    x: [T, H, d] values (bf16 values held in fp64).  For each document, each
    head and each document-local block of ``block`` consecutive tokens (32 by
    default; 1 for the strict per-token option of [EN] section 4): amax over the
    block x head dim, e by the round-up rule, codes = E4M3(x * 2**-e) and one
    UE8M0 byte (e + 127) stored for every token of the block.

    Tokens outside every document keep code 0 and byte 127.
    Returns (codes uint8 [T,H,d], scale bytes uint8 [T,H])."""
    x = np.asarray(x, dtype=np.float64)
    T, H, d = x.shape
    codes = np.zeros((T, H, d), dtype=np.uint8)
    sbytes = np.full((T, H), 127, dtype=np.uint8)
    exp_rule = roundup_exponent if rule == "roundup" else floor_exponent
    for b0, b1 in _doc_blocks(cu, block):
        xb = x[b0:b1]
        amax = np.abs(xb).max(axis=(0, 2))
        e = exp_rule(amax)
        codes[b0:b1] = e4m3_encode(xb * np.ldexp(1.0, -e)[None, :, None])
        sbytes[b0:b1] = (e + 127).astype(np.uint8)[None, :]
    return codes, sbytes


def hadamard_norm_log2(d: int) -> int:
    """k = ceil(log2(d) / 2): the rotation is H / 2**k (see :func:`hadamard_rotate`)."""
    return (int(d).bit_length() - 1 + 1) // 2


def hadamard_rotate(x, dtype=np.float32) -> np.ndarray:
    """Rotation of the head dimension, reading C-18 ([EN] section 3 "Rotation,
    range, and the alternative": an orthogonal normalized Hadamard matrix mixes
    the last dimension before rounding, and the exact score is unchanged; [KO]
    section 3.4: fused into the quantizer, on by default at head dim 128).

    Returns x H~ along the last axis with H~ = H / 2**k, H the d x d Sylvester
    Hadamard matrix (entries +-1, H H = d I) and k = ceil(log2(d) / 2), so the
    scale is a power of two (d = 64: H~ is orthonormal; d = 128: H~ H~ = I / 2).
    It is computed by the fast Walsh-Hadamard butterfly network: for strides
    1, 2, ..., d/2 in increasing order every pair (i, i + stride) with that bit
    of i clear becomes (a + b, a - b), each sum rounded to ``dtype`` (fp32 for
    the quantized route: the codes of the rotated values are bit-exact); then
    the power of two.  H~ is symmetric, so the same map undoes a rotation up to
    the factor d / 4**k."""
    y = np.asarray(x, np.float64).astype(dtype)
    d = y.shape[-1]
    lead = y.shape[:-1]
    st = 1
    while st < d:
        v = y.reshape(lead + (d // (2 * st), 2, st))
        a, b = v[..., 0, :], v[..., 1, :]
        y = np.stack([a + b, a - b], axis=-2).reshape(lead + (d,))
        st *= 2
    return (y * dtype(2.0 ** -hadamard_norm_log2(d))).astype(np.float64)


def dequantize_tokenblock(codes, sbytes) -> np.ndarray:
    """X^ = s_X * c_X with s_X = 2**(byte - 127) per token and head."""
    return e4m3_decode(codes) * ue8m0_decode(sbytes)[:, :, None]


def quantize_nvfp4(x):
    """NVFP4 score operand ([EN] section 2; [KO] section 3.1), reading C-7: no
    tensor scale; per (token, head, 16 head-dim elements) the scale is
    E4M3(amax / 6) computed with an fp32 division and raised to 2**-9 when it
    would round to zero for a non-zero group; codes are E2M1(fp32(x) / s) with
    an IEEE fp32 division.  Returns (codes uint8 [T,H,d] one per byte,
    scale bytes uint8 [T,H,d/16] as E4M3 codes)."""
    x = np.asarray(x, dtype=np.float64)
    T, H, d = x.shape
    g = x.reshape(T, H, d // 16, 16)
    amax = np.abs(g).max(axis=-1).astype(np.float32)
    s = e4m3_round((amax / np.float32(6.0)).astype(np.float64))
    s = np.where((amax > 0) & (s == 0), 2.0 ** -9, s)
    s32 = s.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(s32[..., None] > 0, g.astype(np.float32) / s32[..., None], np.float32(0))
    codes = e2m1_encode(q.astype(np.float64)).reshape(T, H, d)
    return codes, e4m3_encode(s)


def dequantize_nvfp4(codes, scodes) -> np.ndarray:
    T, H, d = codes.shape
    v = e2m1_decode(codes).reshape(T, H, d // 16, 16) * e4m3_decode(scodes)[..., None]
    return v.reshape(T, H, d)


# --------------------------------------------------------------------------
# Cost model and work list.  [EN] section 6 "Cost-based scheduling and tail
# behavior" and Algorithm 2.
# --------------------------------------------------------------------------

def visible_pairs(lengths, window=(-1, 0)) -> int:
    """Visible (query, key) pairs of packed documents: sum n(n+1)/2 for causal
    calls; under a (left, right) window (see :func:`visible_keys`) the sum over
    every query row of the length of its visible key range."""
    if tuple(window) == (-1, 0):
        return int(sum(int(n) * (int(n) + 1) // 2 for n in lengths))
    total = 0
    for n in lengths:
        i = np.arange(int(n))
        lo, hi = visible_keys(i, int(n), window)
        total += int(np.maximum(hi - lo + 1, 0).sum())
    return total


def visible_keys(i, L: int, window=(-1, 0)):
    """Document-local key range [lo, hi] that query i of a document of length L
    sees.  window = (left, right): key j is visible iff i - left <= j <= i + right,
    a negative bound meaning no limit on that side.  Causal calls use (-1, 0)
    (keys up to the query), noncausal calls (-1, -1) (the whole document) --
    the packed noncausal calls of [EN] section 8 / Appendix H; other values give
    sliding windows.  Keys never leave the document."""
    left, right = window
    i = np.asarray(i)
    lo = np.zeros_like(i) if left < 0 else np.maximum(i - left, 0)
    hi = np.full_like(i, L - 1) if right < 0 else np.minimum(i + right, L - 1)
    return lo, hi


def key_tiles(t: int, L: int, window=(-1, 0), tile: int = 128) -> range:
    """Key tiles holding a key that some query of query tile t sees: the rows'
    ranges are consecutive, so their union runs from the first row's lo to the
    last row's hi."""
    first, last = t * tile, min(t * tile + tile, L) - 1
    lo, _ = visible_keys(first, L, window)
    _, hi = visible_keys(last, L, window)
    return range(int(lo) // tile, int(hi) // tile + 1)


def query_tiles(u: int, L: int, window=(-1, 0), tile: int = 128) -> range:
    """Query tiles holding a query that sees some key of key tile u (query i sees
    key j iff j - right <= i <= j + left)."""
    left, right = window
    first, last = u * tile, min(u * tile + tile, L) - 1
    lo = 0 if right < 0 else max(first - right, 0)
    hi = L - 1 if left < 0 else min(last + left, L - 1)
    return range(lo // tile, hi // tile + 1)


def work_list(cu, tile: int = 128, item_tiles: int = 2, num_ctas: Optional[int] = None, window=(-1, 0)):
    """Algorithm 2 of [EN] (steps 03-06) with reading C-11: items of up to
    ``item_tiles`` query tiles (256 queries) of one document; cost = number of
    visible key tiles summed over the item's query tiles (causal); sort by
    decreasing cost (ties keep document order, then query order); alternate the
    assignment direction over persistent CTAs on every pass.

    Returns a list of dicts in sorted order with keys doc, tile0, ntiles, cost
    and (when num_ctas is given) cta."""
    items = []
    for n, (s, t) in enumerate(doc_ranges(cu)):
        ntile = -(-(t - s) // tile)
        for t0 in range(0, ntile, item_tiles):
            nt = min(item_tiles, ntile - t0)
            cost = sum(len(key_tiles(tt, t - s, window, tile)) for tt in range(t0, t0 + nt))
            items.append(dict(doc=n, tile0=t0, ntiles=nt, cost=cost))
    order = sorted(range(len(items)), key=lambda i: (-items[i]["cost"], i))
    out = [items[i] for i in order]
    if num_ctas:
        for r, it in enumerate(out):
            p, pos = divmod(r, num_ctas)
            it["cta"] = pos if p % 2 == 0 else num_ctas - 1 - pos
    return out


def bwd_key_tile_list(cu, tile: int = 128, window=(-1, 0)):
    """Backward work ([EN] Algorithm 2 step 12): one item per document-local key
    tile, cost = number of query tiles that see it, sorted by decreasing cost
    (ties keep document order then key order)."""
    items = []
    for n, (s, t) in enumerate(doc_ranges(cu)):
        ntile = -(-(t - s) // tile)
        for u in range(ntile):
            items.append(dict(doc=n, ktile=u, cost=len(query_tiles(u, t - s, window, tile))))
    order = sorted(range(len(items)), key=lambda i: (-items[i]["cost"], i))
    return [items[i] for i in order]


# --------------------------------------------------------------------------
# Attention.  [EN] section 2 (definitions, centred softmax gradient, online
# recurrence), section 5 (Algorithm 1; range budget for probabilities) and
# [KO] section 1.2 (S = QK^T/sqrt(d), P = softmax(S), O = PV and the five
# backward products).
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Options:
    quantized: bool = True         # False: every codec is the identity
    block: int = 32                # operand token-block length (1 = strict per-token)
    strict: bool = False           # strict options: per-token scales folded into the companion
                                   # operand, per-query-row dS exponents, causal dQ boost
    rule: str = "roundup"          # operand exponent rule ("floor" = negative control)
    p_boost_log2: int = 8          # beta = 2**8 for the forward P operand (reading C-4)
    p_lag_log2: int = 0            # tau: how far the retained max may lag (reading C-4)
    bwd_p_boost_log2: int = 8      # backward P operand boost (reading C-6)
    tile: int = 128                # query and key tile (reading C-11)
    dq_headroom_log2: int = 14     # dQ boost target 2**14 (reading C-10)
    mixed: bool = False            # mixed route: NVFP4 score operands, diagonal per-key V (C-7, C-8)
    window: tuple = (-1, 0)        # (left, right) visible-key window: causal (-1, 0), noncausal (-1, -1)
    rotate: bool = False           # Hadamard rotation of Q and K before quantization (reading C-18)


def _masked_scores(Qt, Ku, qpos, kpos, scale, window=(-1, 0)):
    """scale * Q K^T with the keys a query does not see set to -inf (positions of
    one document; see visible_keys)."""
    left, right = window
    S = scale * (Qt @ Ku.T)
    d = kpos[None, :] - qpos[:, None]
    hidden = np.zeros(d.shape, bool)
    if right >= 0:
        hidden |= d > right
    if left >= 0:
        hidden |= d < -left
    return np.where(hidden, -np.inf, S)


def attention_forward(Qh, Kh, Vh, cu, hq: int, hkv: int, scale: Optional[float] = None,
                      opts: Options = Options(), heads: Optional[Iterable[int]] = None,
                      q_tiles: Optional[Dict[int, Iterable[int]]] = None, v_scale=None,
                      score_ops=None, v_diag=None):
    """Forward of Algorithm 1 (steps 04-08) for causal packed documents.

    Qh [T,hq,d], Kh/Vh [T,hkv,d]: reconstructed operands X^ = s*c (or plain
    values when unquantized).  For every document, query head h (kv head
    h // (hq/hkv)) and 128-row document-local query tile, visit the visible
    128-key tiles in increasing order:

      S   = scale * Q^ K^T, keys after the query masked to -inf
      m'  = max(m, rowmax S)      (retained max may lag by tau, reading C-4)
      p   = exp(S - m'),  l = l * exp(m - m') + sum(p)     (unrounded, C-5)
      P^  = E4M3(beta * p) / beta                          (section 5)
      acc = acc * exp(m - m') + P^ V^

    and finish with O = bf16(acc / l), LSE = m + ln l ([EN] section 2 "Why
    flash tiling recomputes scores").  Rows outside every document keep O = 0
    and LSE = +inf ([EN] section 6).

    Strict options ([EN] section 4, "Folding a local scale into the companion
    operand"; reading in the design notes): operands carry per-token scales
    (v_scale [T, hkv] for V); the per-key V scale is folded into the
    probability operand, P~_ij = beta p_ij s_V(j), which is E4M3-rounded with
    one round-up exponent per (query row, document-local 32-key group), and
    multiplies the V codes.

    Mixed route ([EN] section 2, "the mixed route quantizes Q and K again in
    E4M3 for the gradient products"; [KO] section 3.1; readings C-7, C-8):
    score_ops = (Q~, K~), the reconstructed NVFP4 copies, replace Q^ and K^ in
    S.  On the diagonal key tile (the key tile with the query tile's document-
    local index) V is taken per key: v_diag = (V per-token reconstructed
    [T,hkv,d], s_V [T,hkv]); the per-key scale is folded into the probability
    operand exactly as in the strict route.  Other tiles are unchanged.
    Returns (O [T,hq,d], LSE [hq,T])."""
    Qh = np.asarray(Qh, np.float64); Kh = np.asarray(Kh, np.float64); Vh = np.asarray(Vh, np.float64)
    Qs, Ks = (Qh, Kh) if score_ops is None else (np.asarray(x, np.float64) for x in score_ops)
    T, _, d = Qh.shape
    g = hq // hkv
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    tile = opts.tile
    beta = 2.0 ** opts.p_boost_log2
    tau_nat = opts.p_lag_log2 * math.log(2.0)
    O = np.zeros((T, hq, d))
    LSE = np.full((hq, T), np.inf)
    heads = range(hq) if heads is None else heads
    V_scale = np.asarray(v_scale, np.float64) if opts.strict else None   # [T, hkv] powers of two
    for n, (s0, s1) in enumerate(doc_ranges(cu)):
        ntile = -(-(s1 - s0) // tile)
        tiles = range(ntile) if q_tiles is None else q_tiles.get(n, ())
        for h in heads:
            hk = h // g
            for t in tiles:
                r0, r1 = s0 + t * tile, min(s0 + (t + 1) * tile, s1)
                qpos = np.arange(r0, r1)
                Qt = Qs[r0:r1, h]
                m = np.full(r1 - r0, -np.inf)
                l = np.zeros(r1 - r0)
                acc = np.zeros((r1 - r0, d))
                for u in key_tiles(t, s1 - s0, opts.window, tile):
                    c0, c1 = s0 + u * tile, min(s0 + (u + 1) * tile, s1)
                    S = _masked_scores(Qt, Ks[c0:c1, hk], qpos, np.arange(c0, c1), scale, opts.window)
                    rowmax = S.max(axis=1)
                    m_new = np.where(rowmax > m + tau_nat, np.maximum(m, rowmax), m)
                    with np.errstate(invalid="ignore"):
                        alpha = np.where(np.isfinite(m), np.exp(m - m_new), 0.0)
                    with np.errstate(invalid="ignore"):   # rows that have seen no key yet: p = 0
                        p = np.where(np.isfinite(S), np.exp(S - m_new[:, None]), 0.0)
                    l = l * alpha + p.sum(axis=1)
                    Vt = Vh[c0:c1, hk]
                    if not opts.quantized:
                        Pq = p
                    elif opts.strict or (opts.mixed and u == t):
                        # per-key V scale folded into P, quantized with one round-up exponent
                        # per (query row, document-local 32-key group)
                        if opts.strict:
                            sv = V_scale[c0:c1, hk]
                        else:
                            Vt = np.asarray(v_diag[0], np.float64)[c0:c1, hk]
                            sv = np.asarray(v_diag[1], np.float64)[c0:c1, hk]
                        Pq = _fold_quantize(beta * p * sv[None, :], group_axis=1, offset=c0 - s0) / (beta * sv[None, :])
                    else:
                        Pq = e4m3_round(beta * p) / beta
                    acc = acc * alpha[:, None] + Pq @ Vt
                    m = m_new
                out = acc / l[:, None]
                O[r0:r1, h] = bf16_round(out) if opts.quantized else out
                LSE[h, r0:r1] = m + np.log(l)
    return O, LSE


def dq_boost(dOh_doc, Vh_doc, Kh_doc, headroom_log2: int = 14) -> float:
    """Default dQ accumulator boost for one (document, query head), reading
    C-10 of [EN] section 4 "Forward locality and backward locality differ":
    M = 2 * max_i ||dO^_i|| * max_j ||V^_j|| * max_{j,d} |K^_jd| bounds every
    partial |sum_j dS_ij K_jd|; c = 2**floor(log2(2**14 / M)); c = 1 if M = 0."""
    M = 2.0 * np.sqrt((dOh_doc ** 2).sum(-1)).max(initial=0.0) \
        * np.sqrt((Vh_doc ** 2).sum(-1)).max(initial=0.0) * np.abs(Kh_doc).max(initial=0.0)
    if not (M > 0) or not np.isfinite(M):
        return 1.0
    e = math.floor(math.log2(2.0 ** headroom_log2 / M))
    while 2.0 ** e * M > 2.0 ** headroom_log2:
        e -= 1
    while 2.0 ** (e + 1) * M <= 2.0 ** headroom_log2:
        e += 1
    e = max(-100, min(100, e))
    return 2.0 ** e


def attention_backward(Qh, Kh, Vh, O, LSE, dOh, cu, hq: int, hkv: int,
                       scale: Optional[float] = None, opts: Options = Options(),
                       kv_heads: Optional[Iterable[int]] = None,
                       k_tiles: Optional[Dict[int, Iterable[int]]] = None,
                       q_tiles: Optional[Dict[int, Iterable[int]]] = None,
                       diagnostics: bool = False, tok_scales: Optional[dict] = None, score_ops=None,
                       grad_map=None):
    """Backward of Algorithm 1 (steps 09-16).

    dOh: the reconstructed incoming gradient dO^ (encoded once, step 09);
    D_i = dO^_i . O_i with the saved bf16 O ([KO] section 3.3).  For every
    document, kv head, document-local 128-key tile u (increasing) and every
    query tile t >= u of each query head sharing the kv head:

      S   = scale * Q^ K^T (same tiles and masks as the forward)
      P   = exp(S - LSE)                                  (step 12)
      dP  = dO^ V^T,  dS = P o (dP - D)                   (steps 13-14)
      dS^ = per document-local 32x32 block: E4M3(dS * 2**-e) * 2**e with
            e the round-up exponent of the block amax     (reading C-9)
      dV += (E4M3(2**8 P) / 2**8)^T dO^                  (reading C-6)
      dK += dS^^T Q^
      h   = fp16(c * dS^ K^),  accQ = fp16(accQ + h)      (step 15)

    then dK = bf16(scale * dK), dV = bf16(dV), dQ = bf16(scale * accQ / c)
    (step 16).  Unquantized: every codec is the identity and accQ is exact.

    Strict options (tok_scales = per-token powers of two of q, k, do): the
    per-token scale of the contraction-axis operand is folded into its
    companion, which is E4M3-rounded with one round-up exponent per (row of the
    companion, document-local 32-token group): dV uses beta P s_dO(i) per (key,
    32-query group); dK uses dS s_Q(i) per (key, 32-query group); dQ uses
    dS s_K(j) per (query row, 32-key block) -- the per-query-row dS exponent
    ("K fold").  The dQ boost is the causal per-row c_i (causal_dq_boost).

    Mixed route: score_ops = (Q~, K~) (NVFP4 copies) replace Q^ and K^ in the
    recomputed S only -- the same scores as the forward; every gradient product
    uses the E4M3 copies as in the default route.

    k_tiles / q_tiles restrict which dK/dV key tiles and dQ query tiles are
    produced (others stay zero); kv_heads restricts heads.  grad_map (rotated
    operands): applied along the head dimension to scale * accQ / c and to
    scale * dK before the bf16 rounding, to bring them back to the caller's
    basis.
    Returns dict with dq, dk, dv (and diagnostics when asked)."""
    Qh = np.asarray(Qh, np.float64); Kh = np.asarray(Kh, np.float64)
    Vh = np.asarray(Vh, np.float64); dOh = np.asarray(dOh, np.float64)
    O = np.asarray(O, np.float64); LSE = np.asarray(LSE, np.float64)
    Qs, Ks = (Qh, Kh) if score_ops is None else (np.asarray(x, np.float64) for x in score_ops)
    T, _, d = Qh.shape
    g = hq // hkv
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    tile = opts.tile
    q = opts.quantized
    beta_b = 2.0 ** opts.bwd_p_boost_log2
    D = (dOh * O).sum(-1)                                   # [T, hq]
    dQ = np.zeros((T, hq, d)); dK = np.zeros((T, hkv, d)); dV = np.zeros((T, hkv, d))
    diag = dict(rowsum_ds=np.zeros((hq, T)), rowmax_ds=np.zeros((hq, T)),
                rowsum_p=np.zeros((hq, T)), rowsum_pdp=np.zeros((hq, T)),
                ds_nonzero=0, dsq_zero=0) if diagnostics else None
    if diagnostics and T <= 2048:      # every pair's P and dS before quantization, [hq, query, key]
        diag["p_full"] = np.zeros((hq, T, T))
        diag["ds_full"] = np.zeros((hq, T, T))
    kv_heads = range(hkv) if kv_heads is None else kv_heads
    if opts.strict:   # per-token scales s_X = 2**e of the strict per-token quantization
        Q_scale, K_scale, dO_scale = (np.asarray(tok_scales[n], np.float64) for n in ("q", "k", "do"))
    for n, (s0, s1) in enumerate(doc_ranges(cu)):
        ntile = -(-(s1 - s0) // tile)
        ksel = set(range(ntile)) if k_tiles is None else set(k_tiles.get(n, ()))
        qsel = set(range(ntile)) if q_tiles is None else set(q_tiles.get(n, ()))
        for hk in kv_heads:
            for h in range(hk * g, (hk + 1) * g):
                if q and opts.strict:
                    c = causal_dq_boost(dOh[s0:s1, h], Vh[s0:s1, hk], Kh[s0:s1, hk], opts.dq_headroom_log2)
                elif q:
                    c = dq_boost(dOh[s0:s1, h], Vh[s0:s1, hk], Kh[s0:s1, hk], opts.dq_headroom_log2)
                else:
                    c = 1.0
                accQ = {t: np.zeros((min(tile, s1 - s0 - t * tile), d)) for t in qsel}
                for u in range(ntile):
                    c0, c1 = s0 + u * tile, min(s0 + (u + 1) * tile, s1)
                    kpos = np.arange(c0, c1)
                    for t in query_tiles(u, s1 - s0, opts.window, tile):
                        if u not in ksel and t not in qsel and not diagnostics:
                            continue
                        r0, r1 = s0 + t * tile, min(s0 + (t + 1) * tile, s1)
                        qpos = np.arange(r0, r1)
                        S = _masked_scores(Qs[r0:r1, h], Ks[c0:c1, hk], qpos, kpos, scale, opts.window)
                        P = np.exp(S - LSE[h, r0:r1][:, None])
                        dP = dOh[r0:r1, h] @ Vh[c0:c1, hk].T
                        dS = P * (dP - D[r0:r1, h][:, None])
                        if q and opts.strict:
                            # per-token scales folded into the companion operand of each
                            # token-axis product; one round-up exponent per (row of the
                            # result operand, document-local 32-token group)
                            sdo, sq_ = dO_scale[r0:r1, h], Q_scale[r0:r1, h]
                            sk_ = K_scale[c0:c1, hk]
                            Pq = _fold_quantize(beta_b * P * sdo[:, None], group_axis=0, offset=r0 - s0) / \
                                (beta_b * sdo[:, None])                       # dV: fold s_dO into P^T
                            dSk = _fold_quantize(dS * sq_[:, None], group_axis=0, offset=r0 - s0) / sq_[:, None]
                            dSq = _fold_quantize(dS * sk_[None, :], group_axis=1, offset=c0 - s0) / sk_[None, :]
                        elif q:
                            dSq = _quantize_ds_blocks(dS, r0 - s0, c0 - s0)
                            dSk = dSq
                            Pq = e4m3_round(beta_b * P) / beta_b
                        else:
                            dSq = dSk = dS
                            Pq = P
                        if u in ksel:
                            dV[c0:c1, hk] += Pq.T @ dOh[r0:r1, h]
                            dK[c0:c1, hk] += dSk.T @ Qh[r0:r1, h]
                        if t in qsel:
                            part = dSq @ Kh[c0:c1, hk]
                            if q:
                                ct = c[r0 - s0:r1 - s0, None] if np.ndim(c) else c
                                accQ[t] = fp16_round(accQ[t] + fp16_round(ct * part))
                            else:
                                accQ[t] = accQ[t] + part
                        if diagnostics:
                            diag["rowsum_ds"][h, r0:r1] += dS.sum(1)
                            diag["rowmax_ds"][h, r0:r1] = np.maximum(diag["rowmax_ds"][h, r0:r1],
                                                                     np.abs(dS).max(1))
                            diag["rowsum_p"][h, r0:r1] += P.sum(1)
                            diag["rowsum_pdp"][h, r0:r1] += (P * dP).sum(1)
                            if "p_full" in diag:
                                diag["p_full"][h, r0:r1, c0:c1] = P
                                diag["ds_full"][h, r0:r1, c0:c1] = dS
                            if q:
                                nz = dS != 0
                                diag["ds_nonzero"] += int(nz.sum())
                                diag["dsq_zero"] += int((nz & (dSq == 0)).sum())
                for t in qsel:
                    r0, r1 = s0 + t * tile, min(s0 + (t + 1) * tile, s1)
                    ct = c[r0 - s0:r1 - s0, None] if np.ndim(c) else c
                    dQ[r0:r1, h] = scale * accQ[t] / ct
    dK = scale * dK
    if grad_map is not None:
        dQ, dK = grad_map(dQ), grad_map(dK)
    out = dict(dq=bf16_round(dQ) if q else dQ,
               dk=bf16_round(dK) if q else dK,
               dv=bf16_round(dV) if q else dV)
    if diagnostics:
        out["diag"] = diag
    return out


def _fold_quantize(X, group_axis: int, offset: int, group: int = 32):
    """E4M3 with one round-up exponent per (line, 32-element group along
    group_axis); groups are document-local (offset = document-local index of
    the first element along group_axis, a multiple of 32).  Zero groups take
    exponent 0.  Returns the reconstructed values."""
    assert offset % group == 0
    Xm = np.moveaxis(np.asarray(X, np.float64), group_axis, -1)
    n = Xm.shape[-1]
    npad = -(-n // group) * group
    pad = np.zeros(Xm.shape[:-1] + (npad,))
    pad[..., :n] = Xm
    g = pad.reshape(Xm.shape[:-1] + (npad // group, group))
    e = roundup_exponent(np.abs(g).max(axis=-1))
    sc = np.ldexp(1.0, e)[..., None]
    out = (e4m3_round(g / sc) * sc).reshape(pad.shape)[..., :n]
    return np.moveaxis(out, -1, group_axis)


def causal_dq_boost(dOh_doc, Vh_doc, Kh_doc, headroom_log2: int = 14):
    """Strict causal dQ boost ([EN] section 4, "the causal accumulator scale
    combines ||dO_i|| with running maxima of key and value magnitudes"), reading
    C-10: M_i = 2 ||dO^_i|| max_{j<=i} ||V^_j|| max_{j<=i,d} |K^_jd| and
    c_i = 2**floor(log2(2**14 / M_i)) (1 where M_i = 0).  Returns c per row."""
    a = np.sqrt((dOh_doc ** 2).sum(-1))
    b = np.maximum.accumulate(np.sqrt((Vh_doc ** 2).sum(-1)))
    k = np.maximum.accumulate(np.abs(Kh_doc).max(-1))
    M = 2.0 * a * b * k
    out = np.ones_like(M)
    for i, m in enumerate(M):
        if m > 0 and np.isfinite(m):
            e = math.floor(math.log2(2.0 ** headroom_log2 / m))
            while 2.0 ** e * m > 2.0 ** headroom_log2:
                e -= 1
            while 2.0 ** (e + 1) * m <= 2.0 ** headroom_log2:
                e += 1
            out[i] = 2.0 ** max(-100, min(100, e))
    return out


def _quantize_ds_blocks(dS, qoff: int, koff: int, block: int = 32):
    """Reading C-9: one round-up exponent per document-local 32x32 block of dS
    ([EN] section 3, "the analogous region is a 32 by 32 square"; section 5
    "The paper's 32 by 32 maxima"; [KO] section 3.3).  qoff/koff are the
    document-local offsets of the tile's first row/column (multiples of 32)."""
    R, C = dS.shape
    assert qoff % block == 0 and koff % block == 0
    Rp, Cp = -(-R // block) * block, -(-C // block) * block
    pad = np.zeros((Rp, Cp))
    pad[:R, :C] = dS
    blocks = pad.reshape(Rp // block, block, Cp // block, block)
    e = roundup_exponent(np.abs(blocks).max(axis=(1, 3)))          # [Rb, Cb]
    sc = np.ldexp(1.0, e)[:, None, :, None]
    q = e4m3_round(blocks / sc) * sc
    return q.reshape(Rp, Cp)[:R, :C]


# --------------------------------------------------------------------------
# Brute-force references (textbook definitions, no tiling).  [KO] section
# 1.2; [EN] section 2 "The contraction moves between forward and backward".
# --------------------------------------------------------------------------

def dense_attention(Q, K, V, cu, hq: int, hkv: int, scale: Optional[float] = None, window=(-1, 0)):
    """Masked softmax attention per document and head, whole score matrix at once.
    Returns (O [T,hq,d], LSE [hq,T])."""
    Q = np.asarray(Q, np.float64); K = np.asarray(K, np.float64); V = np.asarray(V, np.float64)
    T, _, d = Q.shape
    g = hq // hkv
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    O = np.zeros((T, hq, d)); LSE = np.full((hq, T), np.inf)
    for s0, s1 in doc_ranges(cu):
        pos = np.arange(s0, s1)
        for h in range(hq):
            S = _masked_scores(Q[s0:s1, h], K[s0:s1, h // g], pos, pos, scale, window)
            mx = S.max(1, keepdims=True)
            E = np.exp(S - mx)
            Z = E.sum(1, keepdims=True)
            O[s0:s1, h] = (E / Z) @ V[s0:s1, h // g]
            LSE[h, s0:s1] = (mx + np.log(Z))[:, 0]
    return O, LSE


def dense_attention_grads(Q, K, V, dO, cu, hq: int, hkv: int, scale: Optional[float] = None, window=(-1, 0)):
    """Textbook gradients: dV = P^T dO, dP = dO V^T, D_i = sum_j P_ij dP_ij,
    dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q (GQA: summed over the
    query heads of a kv head).  Returns dict dq, dk, dv, ds_rowsum [hq,T]."""
    Q = np.asarray(Q, np.float64); K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64); dO = np.asarray(dO, np.float64)
    T, _, d = Q.shape
    g = hq // hkv
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dQ = np.zeros_like(Q); dK = np.zeros_like(K); dV = np.zeros_like(V)
    rows = np.zeros((hq, T))
    for s0, s1 in doc_ranges(cu):
        pos = np.arange(s0, s1)
        for h in range(hq):
            hk = h // g
            S = _masked_scores(Q[s0:s1, h], K[s0:s1, hk], pos, pos, scale, window)
            P = np.exp(S - S.max(1, keepdims=True))
            P /= P.sum(1, keepdims=True)
            dP = dO[s0:s1, h] @ V[s0:s1, hk].T
            Dv = (P * dP).sum(1, keepdims=True)
            dS = P * (dP - Dv)
            rows[h, s0:s1] = dS.sum(1)
            dV[s0:s1, hk] += P.T @ dO[s0:s1, h]
            dQ[s0:s1, h] = scale * dS @ K[s0:s1, hk]
            dK[s0:s1, hk] += scale * dS.T @ Q[s0:s1, h]
    return dict(dq=dQ, dk=dK, dv=dV, ds_rowsum=rows)


# --------------------------------------------------------------------------
# The training call: quantize Q, K, V; forward; encode dO; backward.
# --------------------------------------------------------------------------

def run_training_call(q, k, v, do, cu, hq: int, hkv: int, scale: Optional[float] = None,
                      opts: Options = Options(), **sel):
    """Quantize (Algorithm 1 steps 02-03), forward (04-08), encode dO (09) and
    backward (10-16).  Inputs are bf16 values as fp64 arrays.  ``sel`` may hold
    heads / q_tiles for the forward and kv_heads / k_tiles / bwd_q_tiles for the
    backward (sampled parity at large sizes).  Returns a dict with the codes,
    scale bytes, O, LSE, dq, dk, dv."""
    out = {}
    if opts.rotate:
        if opts.strict or opts.mixed:
            raise ValueError("the rotation is built for the MXFP8 route")
        # Q and K are rotated per token before quantization (Algorithm 1 step 02); the
        # same codes serve the scores and the gradient products; the score scale takes the
        # rotation's d / 4**k, and dQ, dK are rotated back by the same map
        dt = np.float32 if opts.quantized else np.float64
        d = np.asarray(q).shape[-1]
        q, k = hadamard_rotate(q, dt), hadamard_rotate(k, dt)
        out["q_rot"], out["k_rot"] = q, k
        scale = (1.0 / math.sqrt(d) if scale is None else float(scale)) * 4.0 ** hadamard_norm_log2(d) / d
        sel = dict(sel, grad_map=lambda y: hadamard_rotate(y, np.float64))
    if opts.strict and opts.mixed:
        raise ValueError("the strict options and the mixed route are separate configurations")
    if (opts.strict or opts.mixed) and tuple(opts.window) != (-1, 0):
        raise ValueError("the strict options and the mixed route are causal")
    if opts.quantized:
        blk = 1 if opts.strict else opts.block
        for name, x in (("q", q), ("k", k), ("v", v), ("do", do)):
            if x is None:
                continue
            c, sb = quantize_tokenblock(x, cu, blk, opts.rule)
            out[name + "_codes"], out[name + "_scales"] = c, sb
            out[name + "_hat"] = dequantize_tokenblock(c, sb)
    else:
        for name, x in (("q", q), ("k", k), ("v", v), ("do", do)):
            out[name + "_hat"] = np.asarray(x, np.float64)
    tok = {n: ue8m0_decode(out[n + "_scales"]) for n in ("q", "k", "v", "do") if n + "_scales" in out} \
        if opts.quantized else {}
    score_ops = v_diag = None
    if opts.mixed:
        if opts.quantized:
            for name, x in (("q", q), ("k", k)):
                c, sc = quantize_nvfp4(x)
                out[name + "_nvfp4_codes"], out[name + "_nvfp4_scales"] = c, sc
                out[name + "_nvfp4_hat"] = dequantize_nvfp4(c, sc)
            c, sb = quantize_tokenblock(v, cu, 1, opts.rule)          # per-key V for diagonal tiles
            out["v_tok_codes"], out["v_tok_scales"] = c, sb
            out["v_tok_hat"] = dequantize_tokenblock(c, sb)
            score_ops = (out["q_nvfp4_hat"], out["k_nvfp4_hat"])
            v_diag = (out["v_tok_hat"], ue8m0_decode(sb))
        else:
            v_diag = (out["v_hat"], np.ones(np.asarray(v).shape[:2]))
    O, LSE = attention_forward(out["q_hat"], out["k_hat"], out["v_hat"], cu, hq, hkv, scale, opts,
                               heads=sel.get("heads"), q_tiles=sel.get("q_tiles"), v_scale=tok.get("v"),
                               score_ops=score_ops, v_diag=v_diag)
    out["o"], out["lse"] = O, LSE
    if do is not None:
        g = attention_backward(out["q_hat"], out["k_hat"], out["v_hat"], O, LSE, out["do_hat"], cu,
                               hq, hkv, scale, opts, kv_heads=sel.get("kv_heads"),
                               k_tiles=sel.get("k_tiles"), q_tiles=sel.get("bwd_q_tiles"),
                               diagnostics=sel.get("diagnostics", False), tok_scales=tok,
                               score_ops=score_ops, grad_map=sel.get("grad_map"))
        out.update(g)
    return out
