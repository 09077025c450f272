"""Pins for the precision points of the oracle's one-layer step.

``layer_step`` rounds to the activation type at fixed places ("GPU Kernel Lab"
README, "Fundamental kernels" and "Decode integration": the decode step stores
bf16 activations between kernels; the Q8_0 model keeps binary32 activations):
the two RMSNorm casts, the K/V cache write (always bf16), the attention output
that feeds the O projection, and the SwiGLU product that feeds the down
projection. Each scenario below builds a layer from hand-chosen weights so that
exactly one of those points decides one output value, and that value is worked
out by hand (a power-of-two sum or a hand-rounded fraction). Dropping a
rounding, moving it, or using the wrong rounding rule changes the value.

``round_f32`` is pinned against Python's ``struct`` binary32 conversion, a
route that does not go through NumPy.
"""
import math
import struct

import numpy as np
import pytest

import oracle

H, HQ, HKV, D, F = 256, 4, 2, 128, 64
QKV = (HQ + 2 * HKV) * D


def f32_struct(x: float) -> float:
    """IEEE binary32 round-to-nearest-even of a double, through the C library."""
    return struct.unpack("<f", struct.pack("<f", x))[0]


# ---------------------------------------------------------------- round_f32


def test_round_f32_hand_cases():
    # 1 + 2^-24 is halfway between 1 and 1 + 2^-23: ties to even -> 1
    # 1 + 3 * 2^-24 is halfway between 1 + 2^-23 and 1 + 2^-22: ties to even -> 1 + 2^-22
    # 1/3 = 0x3EAAAAAB in binary32 = 11184811 / 2^25
    vals = [1 + 2**-24, 1 + 3 * 2**-24, 1 / 3, -(1 + 2**-24), 2**-149, 2**-150 * 3]
    want = [1.0, 1 + 2**-22, 11184811 / 2**25, -1.0, 2**-149, 2**-148]
    assert list(oracle.round_f32(np.array(vals))) == want


def test_round_f32_matches_struct_conversion():
    rng = np.random.default_rng(21)
    x = rng.standard_normal(20000) * 10.0 ** rng.integers(-40, 38, 20000)
    got = oracle.round_f32(x)
    ref = np.array([f32_struct(float(v)) for v in x])
    np.testing.assert_array_equal(got, ref)


def test_round_f32_rmsnorm_points():
    # f32 mode rounds x * rsqrt(ms + eps) and then w * that, each to binary32
    x = np.ones(64)
    w = oracle.bf16_to_f64(oracle.f64_to_bf16_bits(np.full(64, 1.1)))
    y = oracle.rmsnorm(x, w, 1e-6, mode="f32")
    n = f32_struct(1.0 / math.sqrt(1.0 + 1e-6))
    assert np.all(y == f32_struct(float(w[0]) * n))


# ---------------------------------------------------------------- layer scenarios


def _bf16(a):
    return oracle.f64_to_bf16_bits(np.asarray(a, dtype=np.float64))


def _q8(design_q, design_d):
    """Q8_0 storage from integer codes [R, K] and per-block fp16 scales [R, K/32]."""
    q = np.asarray(design_q, dtype=np.int64)
    assert np.all(np.abs(q) <= 127)
    return q.astype(np.int8), np.asarray(design_d, dtype=np.float64).astype(np.float16).view(np.uint16)


def _bf16_layer(w_qkv, w_o, w_gu, w_down):
    ones_h, ones_d = _bf16(np.ones(H)), _bf16(np.ones(D))
    return oracle.LayerWeights(w_qkv=_bf16(w_qkv), w_o=_bf16(w_o), w_gu=_bf16(w_gu), w_down=_bf16(w_down),
                               ln_in=ones_h, ln_post=ones_h, q_norm=ones_d, k_norm=ones_d)


def _finite_qk(w_qkv):
    """q and k rows that read column 0 (a non-zero head vector, finite under eps = 0)."""
    for h in range(HQ + HKV):
        w_qkv[h * D, 0] = 1.0


def _caches(pos):
    return np.zeros((HKV, pos + 1, D)), np.zeros((HKV, pos + 1, D))


def _attention_output_layer():
    # q = 0 (W_q = 0): all scores 0, so three visible keys get weight 1/3 each.
    # V[0] = 1, V[1] = 0 in the cache, the new token's v = 0 (W_v = 0):
    # o = 1/3 in every head and dimension. W_o row 0 reads o[head 0, dim 0];
    # the MLP adds nothing (W_gu = W_down = 0).
    w_o = np.zeros((H, HQ * D))
    w_o[0, 0] = 1.0
    lw = _bf16_layer(np.zeros((QKV, H)), w_o, np.zeros((2 * F, H)), np.zeros((H, F)))
    kc, vc = _caches(2)
    vc[:, 0, :] = 1.0
    kc[:, :2, :] = 0.5
    return lw, kc, vc


@pytest.mark.parametrize("mode,want", [
    ("bf16", 1 + 171 / 512),          # 1/3 = 1.0101010|10.. b x 2^-2 rounds up to 171/512
    ("f32", 1 + 11184811 / 2**25),    # 1/3 in binary32
    ("exact", 1 + 1 / 3),
])
def test_layer_rounds_the_attention_output(mode, want):
    lw, kc, vc = _attention_output_layer()
    dims = oracle.Dims(H, HQ, HKV, D, F)
    out = oracle.layer_step(dims, lw, np.ones(H), kc, vc, pos=2, mode=mode, act="bf16")
    assert out[0] == want
    np.testing.assert_array_equal(out[1:], 1.0)


def test_layer_rounds_the_attention_output_q8_0_f32_lane():
    # the same scenario with Q8_0 weights on the dequantising lane (f32 activations)
    lw, kc, vc = _attention_output_layer()
    zq = lambda r, c: _q8(np.zeros((r, c)), np.ones((r, c // 32)))  # noqa: E731
    q_o = np.zeros((H, HQ * D))
    q_o[0, 0] = 1
    w_qkv, s_qkv = zq(QKV, H)
    w_o, s_o = _q8(q_o, np.ones((H, HQ * D // 32)))
    w_gu, s_gu = zq(2 * F, H)
    w_dn, s_dn = zq(H, F)
    lq = oracle.LayerWeights(w_qkv, w_o, w_gu, w_dn, lw.ln_in, lw.ln_post, lw.q_norm, lw.k_norm,
                             s_qkv, s_o, s_gu, s_dn)
    out = oracle.layer_step(oracle.Dims(H, HQ, HKV, D, F), lq, np.ones(H), kc, vc, pos=2, mode="f32", act="f32")
    assert out[0] == 1 + 11184811 / 2**25


@pytest.mark.parametrize("mode", ["bf16", "f32", "exact"])
def test_layer_rounds_the_kv_cache_write_to_bf16(mode):
    # eps = 0 and a residual of ones: the normed input is exactly 1 in every lane, so
    # v of kv head 0, dim 0 is 1 + 2^-9 (rounds down to 1 in bf16) and v of kv head 1,
    # dim 3 is 1 + 3 * 2^-9 (rounds up to 1 + 2^-7). The cache holds bf16 in every
    # mode but the exact one.
    w_qkv = np.zeros((QKV, H))
    _finite_qk(w_qkv)
    v0 = (HQ + HKV) * D
    w_qkv[v0 + 0, 0], w_qkv[v0 + 0, 1] = 1.0, 2**-9
    w_qkv[v0 + D + 3, 0], w_qkv[v0 + D + 3, 1] = 1.0, 3 * 2**-9
    lw = _bf16_layer(w_qkv, np.zeros((H, HQ * D)), np.zeros((2 * F, H)), np.zeros((H, F)))
    kc, vc = _caches(5)
    dims = oracle.Dims(H, HQ, HKV, D, F, rms_eps=0.0)
    oracle.layer_step(dims, lw, np.ones(H), kc, vc, pos=5, mode=mode, act="bf16")
    if mode == "exact":
        assert (vc[0, 5, 0], vc[1, 5, 3]) == (1 + 2**-9, 1 + 3 * 2**-9)
    else:
        assert (vc[0, 5, 0], vc[1, 5, 3]) == (1.0, 1 + 2**-7)
        # every K slot value is a bf16 value too
        np.testing.assert_array_equal(oracle.round_bf16(kc[:, 5]), kc[:, 5])
    # q and k read column 0 only: the normed head vector is sqrt(128) e_0, and RoPE at
    # position 5 rotates pair (0, 64) by 5 radians
    r = math.sqrt(128)
    k0, k64 = r * math.cos(5.0), r * math.sin(5.0)
    if mode == "exact":
        assert kc[0, 5, 0] == pytest.approx(k0, rel=1e-15) and kc[0, 5, 64] == pytest.approx(k64, rel=1e-15)
    else:
        assert abs(kc[0, 5, 0] - k0) <= abs(k0) * 2**-8 and abs(kc[0, 5, 64] - k64) <= abs(k64) * 2**-8


def _swiglu_layer(u_small):
    # eps = 0, residual of ones, W_o = 0: the post-attention normed input is exactly 1.
    # gate row 0 = 40 (silu(40) = 40 in binary64), up row 0 = 1 + u_small; W_down row 0
    # reads h[0] = rnd(40 * (1 + u_small)).
    w_qkv = np.zeros((QKV, H))
    _finite_qk(w_qkv)
    w_gu = np.zeros((2 * F, H))
    w_gu[0, 0] = 40.0
    w_gu[F, 0], w_gu[F, 1] = 1.0, u_small
    w_down = np.zeros((H, F))
    w_down[0, 0] = 1.0
    return w_qkv, w_gu, w_down


@pytest.mark.parametrize("u_small,mode,want", [
    (2**-9, "bf16", 41.0),                  # 40.078125 rounds to 40 (bf16 ulp at 40 is 0.25)
    (2**-9, "exact", 41.078125),
    (2**-22, "f32", 41 + 2**-17),           # 40 + 2.5 binary32 ulps: ties to even -> + 2 ulps
    (2**-22, "exact", 41 + 5 * 2**-19),
    (2**-22, "bf16", 41.0),
])
def test_layer_rounds_the_swiglu_product(u_small, mode, want):
    w_qkv, w_gu, w_down = _swiglu_layer(u_small)
    lw = _bf16_layer(w_qkv, np.zeros((H, HQ * D)), w_gu, w_down)
    kc, vc = _caches(3)
    dims = oracle.Dims(H, HQ, HKV, D, F, rms_eps=0.0)
    out = oracle.layer_step(dims, lw, np.ones(H), kc, vc, pos=3, mode=mode, act="bf16")
    assert out[0] == want
    np.testing.assert_array_equal(out[1:], 1.0)


def test_layer_rounds_the_swiglu_product_q8_0_f32_lane():
    # the same scenario in Q8_0 storage: 40 = fp16 1.25 x 32; 2^-22 = fp16 2^-24
    # (the smallest subnormal) x 4 in the second 32-block
    w_qkv, _, _ = _swiglu_layer(2**-22)
    qkv_q = w_qkv.astype(np.int64)
    gu_q, gu_d = np.zeros((2 * F, H)), np.ones((2 * F, H // 32))
    gu_q[0, 0], gu_d[0, 0] = 32, 1.25
    gu_q[F, 0] = 1
    gu_q[F, 32], gu_d[F, 1] = 4, 2.0**-24
    dn_q = np.zeros((H, F))
    dn_q[0, 0] = 1
    ones = np.ones
    w_qkv, s_qkv = _q8(qkv_q, ones((QKV, H // 32)))
    w_o, s_o = _q8(np.zeros((H, HQ * D)), ones((H, HQ * D // 32)))
    w_gu, s_gu = _q8(gu_q, gu_d)
    w_dn, s_dn = _q8(dn_q, ones((H, F // 32)))
    assert oracle.q8_0_dequant(w_gu, s_gu)[F, 32] == 2.0**-22
    n_h, n_d = _bf16(ones(H)), _bf16(ones(D))
    lq = oracle.LayerWeights(w_qkv, w_o, w_gu, w_dn, n_h, n_h, n_d, n_d, s_qkv, s_o, s_gu, s_dn)
    kc, vc = _caches(3)
    out = oracle.layer_step(oracle.Dims(H, HQ, HKV, D, F, rms_eps=0.0), lq, ones(H), kc, vc, pos=3,
                            mode="f32", act="f32")
    assert out[0] == 41 + 2**-17


# ---------------------------------------------------------------- accumulation precision


def test_f32_accumulation_exact_on_integers_and_within_the_summation_bound():
    rng = np.random.default_rng(31)
    # small integers: every partial sum is exact in binary32, so both accumulations agree
    w = rng.integers(-8, 9, size=(40, 512)).astype(np.float64)
    x = rng.integers(-8, 9, size=512).astype(np.float64)
    bits = oracle.f64_to_bf16_bits(w)
    np.testing.assert_array_equal(oracle.gemv_bf16(bits, x, acc="f32"), oracle.gemv_bf16(bits, x))
    ones = np.full((40, 16), 0x3C00, dtype=np.uint16)
    qs = rng.integers(-127, 128, size=(40, 512)).astype(np.int8)
    np.testing.assert_array_equal(oracle.gemv_q8_0(qs, ones, x=x, act="f32", acc="f32"),
                                  oracle.gemv_q8_0(qs, ones, x=x, act="f32"))
    # random bf16 operands: |y32 - y64| <= gamma_(K+1) * sum |w| |x| for any summation
    # order (the classical bound, u = 2^-24), and binary32 is really what is used
    K = 4096
    wb = oracle.f64_to_bf16_bits(rng.standard_normal((64, K)) * 0.02)
    xb = oracle.round_bf16(rng.standard_normal(K))
    y64, y32 = oracle.gemv_bf16(wb, xb), oracle.gemv_bf16(wb, xb, acc="f32")
    u = 2.0 ** -24
    gamma = (K + 1) * u / (1 - (K + 1) * u)
    bound = gamma * (np.abs(oracle.bf16_to_f64(wb)) @ np.abs(xb))
    assert np.all(np.abs(y32 - y64) <= bound)
    assert np.any(y32 != y64)
    np.testing.assert_array_equal(y32, y32.astype(np.float32).astype(np.float64))
    # the dp4a lane: exact integer dots scaled and summed in binary32
    xq, xd = oracle.q8_0_quantize(rng.standard_normal(K).astype(np.float32))
    d = (np.abs(rng.standard_normal((64, K // 32))) * 0.002).astype(np.float16).view(np.uint16)
    q = rng.integers(-127, 128, size=(64, K)).astype(np.int8)
    a64 = oracle.gemv_q8_0(q, d, xq=xq, xd_bits=xd, act="i8")
    a32 = oracle.gemv_q8_0(q, d, xq=xq, xd_bits=xd, act="i8", acc="f32")
    terms = np.abs(oracle.q8_0_block_dots(q, xq) * oracle.f16_to_f64(d) * oracle.f16_to_f64(xd)[None, :]).sum(axis=1)
    nb = K // 32
    assert np.all(np.abs(a32 - a64) <= (nb + 3) * u / (1 - (nb + 3) * u) * terms)
    assert np.any(a32 != a64)


# ---------------------------------------------------------------- INT4 and top-k


def test_int4_unpack_hand_packed_bytes():
    # byte 0x3F: low nibble 15 -> 7, high nibble 3 -> -5; 0x80: 0 -> -8, 8 -> 0
    packed = np.array([[0x3F, 0x80], [0x08, 0xF7]], dtype=np.uint8)
    np.testing.assert_array_equal(oracle.int4_unpack(packed), [[7, -5, -8, 0], [0, -8, -1, 7]])
    d = np.array([0x3C00, 0x4000], dtype=np.uint16)    # fp16 1.0, 2.0
    np.testing.assert_array_equal(oracle.int4_dequant(packed, d), [[7, -5, -8, 0], [0, -16, -2, 14]])


def test_gemv_w4_brute_force_and_unit_scale_exact():
    rng = np.random.default_rng(41)
    R, K = 7, 64
    q = rng.integers(-8, 8, size=(R, K))
    packed = ((q[:, 0::2] + 8) | ((q[:, 1::2] + 8) << 4)).astype(np.uint8)
    x = rng.integers(-9, 10, size=K).astype(np.float64)
    one = np.full(R, 0x3C00, dtype=np.uint16)
    y = oracle.gemv_w4(packed, one, x)
    assert list(y.astype(np.int64)) == [sum(int(q[r, c]) * int(x[c]) for c in range(K)) for r in range(R)]
    d = (np.abs(rng.standard_normal(R)) * 0.01).astype(np.float16)
    xb = oracle.round_bf16(rng.standard_normal(K))
    y = oracle.gemv_w4(packed, d.view(np.uint16), xb)
    for r in range(R):
        ref = math.fsum(float(d[r]) * int(q[r, c]) * float(xb[c]) for c in range(K))
        assert y[r] == pytest.approx(ref, rel=1e-13, abs=1e-15)


def test_topk_first_order_ties_and_nan():
    v = np.array([1.0, 5.0, np.nan, 5.0, -np.inf, 3.0, 5.0])
    idx, val = oracle.topk_first(v, 4)
    assert list(idx) == [1, 3, 6, 5] and list(val) == [5.0, 5.0, 5.0, 3.0]
    idx, _ = oracle.topk_first(np.array([np.nan, -np.inf, -np.inf]), 3)
    assert list(idx) == [1, 2]
    rng = np.random.default_rng(42)
    x = rng.standard_normal(5000)
    idx, _ = oracle.topk_first(x, 8)
    assert idx[0] == oracle.argmax_first(x)
    assert list(idx) == list(np.argsort(-x, kind="stable")[:8])
