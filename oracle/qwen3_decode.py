"""CPU oracle for the Qwen3-style GQA token-decode step.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
arm of ``bench.py`` call it. It shares no code, table or constant generator with
the CUDA library; it receives plain NumPy arrays (bf16 / fp16 storage passed as
raw ``uint16`` bit patterns) from the seeded input generator and computes the
decode math in float64, one obviously-correct step at a time.

Sources (page title, section):
  * "qwen3-8b-rtx4080-cutedsl" README, build-order items "RoPE vectorized kernel",
    "RMSNorm with redux.sync", "GQA + QK-Norm", "Split-KV decode attention".
  * "GPU Kernel Lab" README, "Fundamental kernels" (Qwen-exact RMSNorm cast
    ordering, SwiGLU, RoPE pair rotation, stable softmax) and "Decode
    integration" (the pipeline order of one decode step, argmax + token/position
    update on device).
  * "emit_qwen38_generate" rustdoc, "Where the speed comes from" (concatenated
    projections per shared activation; residual add + next RMSNorm + activation
    re-quantization; the ``deq`` lanes of the Q8_0 GEMV).

Readings where those pages are silent (each also listed in the design notes):
  * RMSNorm: y = w * bf16(x * rsqrt(mean(x^2) + eps)) with the product rounded
    to the activation type (the "Qwen-exact" cast order); eps = 1e-6.
  * RoPE: rotate-half pairing (i, i + D/2), inv_freq_i = theta^(-2i/D),
    angle = pos * inv_freq_i, theta = 1e6, D = 128.
  * QK-norm: per head, before RoPE; no norm on V; the cache holds post-norm,
    post-RoPE K and raw V.
  * Attention: scale 1/sqrt(D), no bias, no mask beyond causality: keys
    0..pos are visible, the current token included; q head h reads kv head
    h // (Hq / Hkv).
  * SwiGLU: silu(g) * u with silu(g) = g / (1 + exp(-g)); the concatenated
    gate+up matrix holds the F gate rows first, then the F up rows.
  * Q8_0: per row, K/32 blocks, w = f32(d) * q with q int8 and d fp16. The
    batched (tensor-core) step widens each weight to bf16 first:
    w = bf16(f32(d) * q), one round-to-nearest-even of the exact product.
    Activation re-quantisation per 32-block: amax = max|x|, d = amax / 127,
    id = 1 / d (0 when d == 0), q = round-half-away-from-zero(x * id), all in
    IEEE binary32, d stored as fp16 (round to nearest even).
  * Argmax: the lowest index among equal maxima; NaN never wins; an all-NaN
    row gives index 0. Top-k: the k largest in that order (value descending,
    lowest index first among equal values), NaN never chosen.
  * INT4 (W4A16, "GPU Kernel Lab" README, "Quantization experiments": W4A16
    decode GEMV, packed INT4 LM head with local top-k, per-output-channel weight
    quantization): q in [-8, 7] with one fp16 scale per output row,
    w = f32(d_r) * q; two values per byte as offset-binary nibbles q + 8, the
    even column in the low nibble. Activations stay bf16.

Accumulation. Every product-sum (the projections) is accumulated in float64
(``acc="f64"``, the default). ``acc="f32"`` evaluates the same sums in IEEE
binary32 instead (operands widened exactly, the library's own summation order).
It is not a model of any kernel: it is a second, equally valid evaluation of the
same rounded computation, used to measure how far a deep bf16 model's outputs move
under ulp-level differences in accumulation alone (the floor any implementation
that does not accumulate in float64 sits on).

Precision modes. ``exact`` computes every step in float64 with no rounding
(used by the closed-form pins). ``bf16`` additionally rounds to bfloat16 at the
points where the bf16 decode step stores a value in bf16: the two RMSNorm
casts, the K/V cache write, the attention output that feeds the O projection
and the SwiGLU product that feeds the down projection. ``f32`` rounds those
points to binary32 instead (the Q8_0 model keeps f32 activations). Everything
between those points stays float64.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# --------------------------------------------------------------------------
# storage formats
# --------------------------------------------------------------------------


def bf16_to_f64(bits) -> np.ndarray:
    """Widen raw bfloat16 bit patterns (uint16) to float64 exactly."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def f16_to_f64(bits) -> np.ndarray:
    """Widen raw IEEE half bit patterns (uint16) to float64 exactly."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round float64 -> binary32 -> bfloat16, each step round-to-nearest-even.

    Returns the uint16 bit patterns. (The decode step rounds binary32 values to
    bf16, so the first rounding to binary32 mirrors where its value lives.)
    """
    u = np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32)
    u = u.astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return u.astype(np.uint16)


def round_bf16(x) -> np.ndarray:
    return bf16_to_f64(f64_to_bf16_bits(x))


def round_f32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def _identity(x):
    return np.asarray(x, dtype=np.float64)


ROUNDERS = {"exact": _identity, "bf16": round_bf16, "f32": round_f32}


# --------------------------------------------------------------------------
# per-op definitions
# --------------------------------------------------------------------------


def rmsnorm(x, w, eps: float = 1e-6, mode: str = "exact") -> np.ndarray:
    """RMSNorm over the last axis, Qwen cast order.

    "GPU Kernel Lab" README, "Fundamental kernels" (Qwen-exact RMSNorm):
    normalise in full precision, cast to the activation type, then multiply by
    the weight and cast again.
    """
    rnd = ROUNDERS[mode]
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    n = rnd(x / np.sqrt(ms + eps))
    return rnd(np.asarray(w, dtype=np.float64) * n)


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    i = np.arange(head_dim // 2, dtype=np.float64)
    return theta ** (-2.0 * i / head_dim)


def rope(x, pos: int, theta: float = 1e6) -> np.ndarray:
    """Rotate-half RoPE over the last axis (pairs (i, i + D/2)).

    "qwen3-8b-rtx4080-cutedsl" README, "RoPE vectorized kernel"; "GPU Kernel
    Lab" README, "Fundamental kernels" (RoPE pair rotation).
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    ang = float(pos) * rope_inv_freq(d, theta)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def softmax(s) -> np.ndarray:
    s = np.asarray(s, dtype=np.float64)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def gqa_attention(q, k, v, scale: float | None = None) -> np.ndarray:
    """Decode attention of one token over T cached keys.

    q: [Hq, D]; k, v: [Hkv, T, D]. q head h reads kv head h // (Hq / Hkv)
    ("qwen3-8b-rtx4080-cutedsl" README, "GQA + QK-Norm"). Split-KV
    (Flash-Decoding, same README, "Split-KV decode attention") only reorders
    this sum, so the oracle is the unsplit softmax.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    hq, d = q.shape
    hkv = k.shape[0]
    rep = hq // hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.empty((hq, d), dtype=np.float64)
    for h in range(hq):
        g = h // rep
        p = softmax(k[g] @ q[h] * scale)
        out[h] = p @ v[g]
    return out


def silu(g) -> np.ndarray:
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def gemv(w, x) -> np.ndarray:
    """y = W x with W [R, K] (float64) and x [K]."""
    return np.asarray(w, dtype=np.float64) @ np.asarray(x, dtype=np.float64)


def _matvec(w, x, acc: str):
    """w @ x with float64 accumulation, or in binary32 (w and x rounded to binary32
    first; exact for bf16 / Q8_0 weights and for bf16 or binary32 activations)."""
    if acc == "f64":
        return w @ x
    if acc == "f32":
        return (np.asarray(w, dtype=np.float32) @ np.asarray(x, dtype=np.float32)).astype(np.float64)
    raise ValueError(acc)


def gemv_bf16(w_bits, x, row_chunk: int = 8192, acc: str = "f64") -> np.ndarray:
    """y = W x with W given as bf16 bits [R, K]; widened a block of rows at a time."""
    w_bits = np.asarray(w_bits)
    x = np.asarray(x, dtype=np.float64)
    r = w_bits.shape[0]
    y = np.empty(r, dtype=np.float64)
    for r0 in range(0, r, row_chunk):
        y[r0:r0 + row_chunk] = _matvec(bf16_to_f64(w_bits[r0:r0 + row_chunk]), x, acc)
    return y


# --------------------------------------------------------------------------
# Q8_0
# --------------------------------------------------------------------------

QK8_0 = 32


def q8_0_dequant(qs, d_bits) -> np.ndarray:
    """W[r, k] = f32(d[r, k // 32]) * q[r, k]."""
    qs = np.asarray(qs, dtype=np.int8).astype(np.float64)
    d = f16_to_f64(d_bits)
    r, k = qs.shape
    return (qs.reshape(r, k // QK8_0, QK8_0) * d[:, :, None]).reshape(r, k)


def q8_0_widen_bf16(qs, d_bits) -> np.ndarray:
    """Each Q8_0 weight rounded once to bfloat16: W[r, k] = bf16(f32(d[r, k // 32]) * q[r, k]).

    The batched projections run on bf16 tensor cores, so each weight is widened
    to bf16 before the contraction. q has at most 8 significant bits and d (fp16)
    at most 11, so the product is exact in binary32 and in float64; the one
    rounding is round-to-nearest-even of the exact product.
    """
    return round_bf16(q8_0_dequant(qs, d_bits))


def q8_0_quantize(x_f32):
    """Per-32-block int8 re-quantisation of a binary32 activation vector.

    Every float step is an IEEE binary32 operation on binary32 inputs, as the
    encoding defines it; only the final round-half-away-from-zero is taken in
    float64, where x * id (a binary32 value) plus 0.5 is exact.
    Returns (q int8 [K], d fp16 bits [K/32]).
    """
    x = np.asarray(x_f32, dtype=np.float32)
    assert x.ndim == 1 and x.size % QK8_0 == 0
    xb = x.reshape(-1, QK8_0)
    amax = np.max(np.abs(xb), axis=1)                      # binary32
    d = (amax / np.float32(127.0)).astype(np.float32)      # binary32 division
    with np.errstate(divide="ignore"):
        idv = np.where(d != 0, np.float32(1.0) / d, np.float32(0.0)).astype(np.float32)
    v = (xb * idv[:, None]).astype(np.float32)             # binary32 multiply
    v64 = v.astype(np.float64)
    q = np.sign(v64) * np.floor(np.abs(v64) + 0.5)
    q = np.clip(q, -127, 127).astype(np.int8)
    d_bits = d.astype(np.float16).view(np.uint16)
    return q.reshape(-1), d_bits


def q8_0_block_dots(qs, xq) -> np.ndarray:
    """Exact integer block dots: D[r, b] = sum_i qs[r, 32b + i] * xq[32b + i]."""
    qs = np.asarray(qs, dtype=np.int8).astype(np.int64)
    xq = np.asarray(xq, dtype=np.int8).astype(np.int64)
    r, k = qs.shape
    return (qs.reshape(r, k // QK8_0, QK8_0) * xq.reshape(1, k // QK8_0, QK8_0)).sum(axis=2)


def gemv_q8_0(qs, d_bits, x=None, xq=None, xd_bits=None, act: str = "f32",
              row_chunk: int = 8192, acc: str = "f64") -> np.ndarray:
    """Q8_0 GEMV, both lanes of the "emit_qwen38_generate" rustdoc's ``deq`` knob.

    act == "f32": y_r = sum_b f32(d_rb) * sum_i q_rbi * x_bi   (dequantising lane)
    act == "i8":  y_r = sum_b f32(d_rb) * f32(dx_b) * sum_i q_rbi * xq_bi  (dp4a lane)
    act == "w_bf16": y_r = sum_k bf16(f32(d_rb) * q_rk) * x_k  (tensor-core lane of the
                  batched step: weights widened to bf16, x the bf16 activation)
    """
    qs = np.asarray(qs, dtype=np.int8)
    r, k = qs.shape
    y = np.empty(r, dtype=np.float64)
    if act == "f32":
        x = np.asarray(x, dtype=np.float64)
        for r0 in range(0, r, row_chunk):
            y[r0:r0 + row_chunk] = _matvec(q8_0_dequant(qs[r0:r0 + row_chunk],
                                                        np.asarray(d_bits)[r0:r0 + row_chunk]), x, acc)
    elif act == "i8":
        dx = f16_to_f64(xd_bits)
        ft = np.float64 if acc == "f64" else np.float32
        for r0 in range(0, r, row_chunk):
            dots = q8_0_block_dots(qs[r0:r0 + row_chunk], xq).astype(ft)
            dw = f16_to_f64(np.asarray(d_bits)[r0:r0 + row_chunk]).astype(ft)
            y[r0:r0 + row_chunk] = (dots * dw * dx.astype(ft)[None, :]).sum(axis=1, dtype=ft)
    elif act == "w_bf16":
        x = np.asarray(x, dtype=np.float64)
        for r0 in range(0, r, row_chunk):
            y[r0:r0 + row_chunk] = _matvec(q8_0_widen_bf16(qs[r0:r0 + row_chunk],
                                                           np.asarray(d_bits)[r0:r0 + row_chunk]), x, acc)
    else:
        raise ValueError(act)
    return y


# --------------------------------------------------------------------------
# INT4 (W4A16)
# --------------------------------------------------------------------------


def int4_unpack(packed) -> np.ndarray:
    """Codes q [R, K] (int64, -8 .. 7) of packed rows [R, K / 2] (uint8)."""
    b = np.asarray(packed, dtype=np.uint8).astype(np.int64)
    r, kh = b.shape
    q = np.empty((r, 2 * kh), dtype=np.int64)
    q[:, 0::2] = (b & 0xF) - 8
    q[:, 1::2] = (b >> 4) - 8
    return q


def int4_dequant(packed, d_bits) -> np.ndarray:
    """W[r, k] = f32(d[r]) * q[r, k]."""
    return int4_unpack(packed).astype(np.float64) * f16_to_f64(d_bits)[:, None]


def gemv_w4(packed, d_bits, x, row_chunk: int = 8192, acc: str = "f64") -> np.ndarray:
    """y = W x for INT4 rows with per-row scales; x is the bf16 activation."""
    packed = np.asarray(packed)
    x = np.asarray(x, dtype=np.float64)
    r = packed.shape[0]
    y = np.empty(r, dtype=np.float64)
    for r0 in range(0, r, row_chunk):
        y[r0:r0 + row_chunk] = _matvec(int4_dequant(packed[r0:r0 + row_chunk], np.asarray(d_bits)[r0:r0 + row_chunk]),
                                       x, acc)
    return y


# --------------------------------------------------------------------------
# argmax, top-k, paged addressing
# --------------------------------------------------------------------------


def topk_first(logits, k: int):
    """The k largest logits, value descending, the lower index first among equal
    values, NaN never chosen: (indices, values). Fewer than k non-NaN entries give
    fewer results."""
    raw = np.asarray(logits, dtype=np.float64)
    idx = np.arange(raw.size)
    ok = ~np.isnan(raw)
    order = np.lexsort((idx[ok], -raw[ok]))   # last key primary: value descending, then index
    sel = idx[ok][order][:k]
    return sel, raw[sel]


def argmax_first(logits) -> int:
    """Lowest index of the maximum; NaN never wins; all-NaN gives 0."""
    raw = np.asarray(logits, dtype=np.float64)
    if raw.size == 0:
        raise ValueError("empty logits")
    nan = np.isnan(raw)
    if nan.all():
        return 0
    a = np.where(nan, -np.inf, raw)
    return int(np.argmax(a))


def paged_token_index(page_table, t: int, page_size: int) -> int:
    """Physical token slot of logical token t: page_table[t // ps] * ps + t % ps."""
    return int(page_table[t // page_size]) * page_size + t % page_size


def gather_paged(pages, page_table, n_tokens: int):
    """Logical [Hkv, T, D] view of a paged cache laid out [pages, Hkv, ps, D]."""
    pages = np.asarray(pages)
    npg, hkv, ps, d = pages.shape
    out = np.empty((hkv, n_tokens, d), dtype=pages.dtype)
    for t in range(n_tokens):
        p = int(page_table[t // ps])
        out[:, t, :] = pages[p, :, t % ps, :]
    return out


# --------------------------------------------------------------------------
# one decoder layer, one token, and the whole model
# --------------------------------------------------------------------------


@dataclass
class Dims:
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6

    @property
    def q_dim(self):
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self):
        return self.n_kv_heads * self.head_dim


@dataclass
class LayerWeights:
    """One layer's weights as NumPy storage arrays.

    BF16 model: ``w_*`` are uint16 bf16 bits [rows, cols] and ``s_*`` are None.
    Q8_0 model: ``w_*`` are int8 [rows, cols] and ``s_*`` uint16 fp16 bits
    [rows, cols / 32]. INT4 model: ``w_*`` are packed uint8 [rows, cols / 2] and
    ``s_*`` uint16 fp16 bits [rows]. Norm weights are uint16 bf16 bits.
    Row order: w_qkv = [q rows (Hq*D); k rows (Hkv*D); v rows (Hkv*D)],
    w_gu = [gate rows (F); up rows (F)].
    """
    w_qkv: np.ndarray
    w_o: np.ndarray
    w_gu: np.ndarray
    w_down: np.ndarray
    ln_in: np.ndarray
    ln_post: np.ndarray
    q_norm: np.ndarray
    k_norm: np.ndarray
    s_qkv: np.ndarray | None = None
    s_o: np.ndarray | None = None
    s_gu: np.ndarray | None = None
    s_down: np.ndarray | None = None


def project(w, s, x, act: str, acc: str = "f64"):
    """One weight-streaming projection for either storage format.

    act == "bf16": W bf16, x already in its storage precision.
    act == "f32":  Q8_0 dequantising lane (x binary32).
    act == "i8":   Q8_0 dp4a lane: x re-quantised per 32-block first.
    act == "w_bf16": Q8_0 weights widened to bf16, x bf16 (batched tensor-core step).
    act == "w4":   INT4 weights with per-row scales (packed uint8, fp16 scales), x bf16.
    """
    if act == "bf16":
        return gemv_bf16(w, x, acc=acc)
    if act == "f32":
        return gemv_q8_0(w, s, x=x, act="f32", acc=acc)
    if act == "i8":
        xq, xd = q8_0_quantize(np.asarray(x, dtype=np.float64).astype(np.float32))
        return gemv_q8_0(w, s, xq=xq, xd_bits=xd, act="i8", acc=acc)
    if act == "w_bf16":
        return gemv_q8_0(w, s, x=x, act="w_bf16", acc=acc)
    if act == "w4":
        return gemv_w4(w, s, x, acc=acc)
    raise ValueError(act)


def layer_step(dims: Dims, lw: LayerWeights, res, k_cache, v_cache, pos: int,
               mode: str = "bf16", act: str = "bf16", trace: dict | None = None, acc: str = "f64"):
    """One decoder layer for one token at position ``pos``.

    Pipeline order from "GPU Kernel Lab" README, "Decode integration":
    projections -> Q/K RMSNorm + RoPE + direct K/V cache write -> GQA
    attention -> attention residual + post-attention RMSNorm -> gate/up GEMV +
    SwiGLU -> down projection + MLP residual.

    res: float64 [H] residual stream (updated copy returned).
    k_cache, v_cache: float64 [Hkv, >= pos+1, D], modified in place at ``pos``.
    """
    rnd = ROUNDERS[mode]
    H, D, hq, hkv, F = dims.hidden, dims.head_dim, dims.n_q_heads, dims.n_kv_heads, dims.ffn
    res = np.asarray(res, dtype=np.float64).copy()
    xn = rmsnorm(res, bf16_to_f64(lw.ln_in), dims.rms_eps, mode)
    qkv = project(lw.w_qkv, lw.s_qkv, xn, act, acc)
    q = qkv[:hq * D].reshape(hq, D)
    k = qkv[hq * D:(hq + hkv) * D].reshape(hkv, D)
    v = qkv[(hq + hkv) * D:].reshape(hkv, D)
    q = rope(rmsnorm(q, bf16_to_f64(lw.q_norm), dims.rms_eps, mode), pos, dims.rope_theta)
    k = rope(rmsnorm(k, bf16_to_f64(lw.k_norm), dims.rms_eps, mode), pos, dims.rope_theta)
    # the cache stores bf16 in every precision mode except "exact"
    kv_rnd = _identity if mode == "exact" else round_bf16
    k_cache[:, pos, :] = kv_rnd(k)
    v_cache[:, pos, :] = kv_rnd(v)
    o = gqa_attention(q, k_cache[:, :pos + 1, :], v_cache[:, :pos + 1, :])
    o = rnd(o.reshape(-1))
    res = res + project(lw.w_o, lw.s_o, o, act, acc)
    xn2 = rmsnorm(res, bf16_to_f64(lw.ln_post), dims.rms_eps, mode)
    gu = project(lw.w_gu, lw.s_gu, xn2, act, acc)
    a = rnd(silu(gu[:F]) * gu[F:])
    res = res + project(lw.w_down, lw.s_down, a, act, acc)
    if trace is not None:
        trace.update(q=q, k=k, v=v, attn=o, xn=xn, xn2=xn2, gu=gu)
    return res


@dataclass
class Model:
    dims: Dims
    layers: list
    embed: np.ndarray            # bf16 bits [V, H]
    final_norm: np.ndarray       # bf16 bits [H]
    lm_head: np.ndarray          # bf16 bits [V, H] or int8 [V, H]
    lm_head_scales: np.ndarray | None = None
    extra: dict = field(default_factory=dict)


def decode_token(model: Model, tok: int, pos: int, k_caches, v_caches,
                 mode: str = "bf16", act: str = "bf16", lm_act: str | None = None,
                 residual_trace: list | None = None, acc: str = "f64"):
    """Logits for one token at position ``pos``; the caches gain slot ``pos``.

    "GPU Kernel Lab" README, "Decode integration": embedding row of the token
    from the fixed token buffer, every layer, the final RMSNorm and the LM-head
    GEMV. ``lm_act`` selects the LM-head lane separately (the ``deq`` = 1 mode
    of the "emit_qwen38_generate" rustdoc keeps only the LM head in f32).
    """
    d = model.dims
    res = bf16_to_f64(model.embed[tok])
    for li, lw in enumerate(model.layers):
        if residual_trace is not None:
            residual_trace.append(res.copy())
        res = layer_step(d, lw, res, k_caches[li], v_caches[li], pos, mode, act, acc=acc)
    if residual_trace is not None:
        residual_trace.append(res.copy())
    xf = rmsnorm(res, bf16_to_f64(model.final_norm), d.rms_eps, mode)
    lm_act = act if lm_act is None else lm_act
    return project(model.lm_head, model.lm_head_scales, xf, lm_act, acc)


def lm_head_rows(model: Model, final_res, rows, mode: str = "bf16", act: str = "bf16"):
    """Selected logits only (sampled parity at full vocabulary size)."""
    d = model.dims
    xf = rmsnorm(np.asarray(final_res, dtype=np.float64), bf16_to_f64(model.final_norm),
                 d.rms_eps, mode)
    rows = np.asarray(rows)
    s = None if model.lm_head_scales is None else np.asarray(model.lm_head_scales)[rows]
    return project(np.asarray(model.lm_head)[rows], s, xf, act)
