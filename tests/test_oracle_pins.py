"""Pins for the CPU oracle: closed forms, invariants, special cases, brute force.

Each test is chosen so a plausible slip in the oracle (a dropped term, a wrong
sign or index, a transposed operand, the wrong rounding rule) fails it. None
retypes the oracle's own formula: the checks go through a different route
(complex multiplication, pure-Python loops, integer arithmetic, hand-worked
values, a library conversion).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- storage


def test_bf16_rounding_matches_hand_values_and_torch():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even -> 1.0 (0x3F80)
    # 1 + 3*2^-8 is halfway between 0x3F81 and 0x3F82: ties to even -> 0x3F82
    vals = np.array([1.0, 1 + 2**-8, 1 + 3 * 2**-8, -2.5, 3.0e38, 1e-40, 0.0, -0.0])
    bits = oracle.f64_to_bf16_bits(vals)
    assert list(bits[:4]) == [0x3F80, 0x3F80, 0x3F82, 0xC020]
    ref = torch.tensor(vals.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, ref)
    rng = np.random.default_rng(0)
    x = rng.standard_normal(10000) * 10.0 ** rng.integers(-30, 30, 10000)
    ref = torch.tensor(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.f64_to_bf16_bits(x), ref)
    # widening is exact and inverse on the representable set
    assert np.array_equal(oracle.f64_to_bf16_bits(oracle.bf16_to_f64(ref)), ref)


# ---------------------------------------------------------------- RMSNorm


def test_rmsnorm_hand_value():
    # x = [3, 4]: mean(x^2) = 12.5; eps = 0: y = x / sqrt(12.5)
    y = oracle.rmsnorm(np.array([3.0, 4.0]), np.ones(2), eps=0.0)
    assert y[0] == pytest.approx(0.8485281374238570, rel=1e-15)
    assert y[1] == pytest.approx(1.1313708498984760, rel=1e-15)


@pytest.mark.parametrize("scale", [1e-4, 1e-2, 1.0, 1e2, 1e4])
def test_rmsnorm_unit_rms_closed_form(scale):
    # unit weight: RMS(y) = 1 / sqrt(1 + eps / mean(x^2)), at any input scale
    rng = np.random.default_rng(1)
    x = rng.standard_normal(4096) * scale
    eps = 1e-6
    y = oracle.rmsnorm(x, np.ones_like(x), eps)
    ms = float(np.dot(x, x)) / x.size
    assert math.sqrt(float(np.dot(y, y)) / y.size) == pytest.approx(1 / math.sqrt(1 + eps / ms), rel=1e-12)


def test_rmsnorm_scale_invariance_and_weight_is_elementwise():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(512)
    w = rng.standard_normal(512)
    y1 = oracle.rmsnorm(x, w, eps=0.0)
    y2 = oracle.rmsnorm(37.5 * x, w, eps=0.0)
    np.testing.assert_allclose(y1, y2, rtol=1e-13)
    # weight multiplies element by element: w = e_j keeps only component j
    e = np.zeros(512)
    e[17] = 1.0
    yj = oracle.rmsnorm(x, e, eps=0.0)
    assert np.count_nonzero(yj) == 1 and yj[17] == pytest.approx(y1[17] / w[17])


def test_rmsnorm_cast_order_bf16():
    # all-ones input: x * rsqrt(1 + 1e-6) = 0.9999995 rounds to 1.0 in bf16, so the
    # Qwen cast order returns the (bf16) weight exactly; the exact mode does not.
    rng = np.random.default_rng(3)
    w = oracle.round_bf16(1 + 0.1 * rng.standard_normal(128))
    y = oracle.rmsnorm(np.ones(128), w, 1e-6, mode="bf16")
    assert np.array_equal(y, w)
    ye = oracle.rmsnorm(np.ones(128), w, 1e-6, mode="exact")
    assert not np.array_equal(ye, w)


# ---------------------------------------------------------------- RoPE


def test_rope_is_complex_rotation():
    # RoPE on pair (i, i + 64) == complex multiply (x_i + i x_{i+64}) * exp(i p theta_i)
    rng = np.random.default_rng(4)
    x = rng.standard_normal(128)
    for pos in (0, 1, 5, 128, 4223):
        y = oracle.rope(x, pos, 1e6)
        z = x[:64] + 1j * x[64:]
        freq = np.array([1e6 ** (-(2 * i) / 128) for i in range(64)])
        w = z * np.exp(1j * pos * freq)
        np.testing.assert_allclose(y[:64], w.real, atol=1e-12)
        np.testing.assert_allclose(y[64:], w.imag, atol=1e-12)


def test_rope_special_values():
    e0 = np.zeros(128)
    e0[0] = 1.0
    y = oracle.rope(e0, 1, 1e6)            # pair 0 has inverse frequency 1
    assert y[0] == pytest.approx(math.cos(1.0), abs=1e-15)
    assert y[64] == pytest.approx(math.sin(1.0), abs=1e-15)
    assert np.count_nonzero(y) == 2
    e1 = np.zeros(128)
    e1[1] = 1.0                              # pair 1: 1e6^(-2/128) = 10^(-6/64)
    y = oracle.rope(e1, 1, 1e6)
    assert y[1] == pytest.approx(math.cos(10 ** (-0.09375)), abs=1e-15)
    assert y[65] == pytest.approx(math.sin(10 ** (-0.09375)), abs=1e-15)
    x = np.arange(128.0)
    np.testing.assert_array_equal(oracle.rope(x, 0), x)   # p = 0 is the identity


def test_rope_norm_and_relativity():
    rng = np.random.default_rng(5)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    for p in (3, 900, 4100):
        y = oracle.rope(q, p)
        pair = lambda v: v[:64] ** 2 + v[64:] ** 2  # noqa: E731
        np.testing.assert_allclose(pair(y), pair(q), rtol=1e-12)
    # <R_p q, R_s k> depends only on p - s
    a = np.dot(oracle.rope(q, 1000), oracle.rope(k, 990))
    b = np.dot(oracle.rope(q, 10), oracle.rope(k, 0))
    assert a == pytest.approx(b, rel=1e-9)


# ---------------------------------------------------------------- attention


def _attn_loop(q, k, v):
    """Direct pure-Python loop: scores, max, exponentials, weighted sum."""
    hq, d = q.shape
    hkv, t, _ = k.shape
    out = np.zeros((hq, d))
    for h in range(hq):
        g = h * hkv // hq
        s = [math.fsum(q[h, j] * k[g, i, j] for j in range(d)) / math.sqrt(d) for i in range(t)]
        m = max(s)
        e = [math.exp(si - m) for si in s]
        z = math.fsum(e)
        for j in range(d):
            out[h, j] = math.fsum(e[i] * v[g, i, j] for i in range(t)) / z
    return out


@pytest.mark.parametrize("hq,hkv,t", [(4, 2, 1), (4, 2, 7), (4, 2, 40), (8, 2, 33), (2, 2, 5)])
def test_attention_brute_force(hq, hkv, t):
    rng = np.random.default_rng(hq * 100 + t)
    q = rng.standard_normal((hq, 128))
    k = rng.standard_normal((hkv, t, 128))
    v = rng.standard_normal((hkv, t, 128))
    np.testing.assert_allclose(oracle.gqa_attention(q, k, v), _attn_loop(q, k, v), rtol=1e-11, atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((8, 128))
    k = rng.standard_normal((2, 50, 128))
    # V == 1 -> output == 1
    np.testing.assert_allclose(oracle.gqa_attention(q, k, np.ones((2, 50, 128))), 1.0, rtol=1e-13)
    # one key -> its value
    v1 = rng.standard_normal((2, 1, 128))
    o = oracle.gqa_attention(q, k[:, :1], v1)
    for h in range(8):
        np.testing.assert_allclose(o[h], v1[h // 4, 0], rtol=1e-13)
    # identical keys -> mean of V
    kk = np.repeat(k[:, :1], 50, axis=1)
    v = rng.standard_normal((2, 50, 128))
    o = oracle.gqa_attention(q, kk, v)
    for h in range(8):
        np.testing.assert_allclose(o[h], v[h // 4].mean(axis=0), rtol=1e-12)
    # GQA grouping: q head h reads kv head h // 4 (not h % 2)
    vc = np.stack([np.full((50, 128), 10.0), np.full((50, 128), -3.0)])
    o = oracle.gqa_attention(q, k, vc)
    assert np.allclose(o[:4], 10.0) and np.allclose(o[4:], -3.0)


def test_softmax_rows_sum_to_one():
    rng = np.random.default_rng(7)
    s = rng.standard_normal((16, 300)) * 50
    np.testing.assert_allclose(oracle.softmax(s).sum(axis=1), 1.0, rtol=1e-14)


def test_silu_special_values():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(1.0) == pytest.approx(1 / (1 + math.exp(-1)), rel=1e-15)
    assert oracle.silu(-40.0) == pytest.approx(-40 * math.exp(-40), rel=1e-10)
    assert oracle.silu(40.0) == pytest.approx(40.0, rel=1e-15)


# ---------------------------------------------------------------- GEMV


def test_gemv_bf16_integer_exact():
    # integer-valued bf16 weights and inputs: exact integer result
    rng = np.random.default_rng(8)
    w = rng.integers(-8, 9, size=(37, 96))
    x = rng.integers(-8, 9, size=96)
    bits = oracle.f64_to_bf16_bits(w.astype(np.float64))
    y = oracle.gemv_bf16(bits, x.astype(np.float64), row_chunk=5)
    ref = [sum(int(w[r, c]) * int(x[c]) for c in range(96)) for r in range(37)]
    assert list(y.astype(np.int64)) == ref


def test_gemv_rank_one():
    rng = np.random.default_rng(9)
    u, v, x = rng.standard_normal(50), rng.standard_normal(64), rng.standard_normal(64)
    y = oracle.gemv(np.outer(u, v), x)
    np.testing.assert_allclose(y, u * np.dot(v, x), rtol=1e-12)


# ---------------------------------------------------------------- Q8_0


def _golden_q8():
    cases, cur = [], {}
    with open(os.path.join(GOLDEN, "q8_0_quantize_hand.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, vals = line.split(":", 1)
            cur[key] = [float(t) for t in vals.split()]
            if key == "d":
                cases.append(cur)
                cur = {}
    return cases


@pytest.mark.parametrize("case", _golden_q8())
def test_q8_0_quantize_hand_cases(case):
    q, d = oracle.q8_0_quantize(np.array(case["x"], dtype=np.float32))
    assert list(q.astype(int)) == [int(v) for v in case["q"]]
    assert oracle.f16_to_f64(d)[0] == case["d"][0]


def test_q8_0_quantize_roundtrip_bound():
    # |x - d*q| <= d/2 (+ binary32 slack) for every element, codes within [-127, 127]
    rng = np.random.default_rng(10)
    x = (rng.standard_normal(4096) * 3).astype(np.float32)
    q, d = oracle.q8_0_quantize(x)
    df = (np.abs(x.reshape(-1, 32)).max(axis=1) / 127).astype(np.float64)
    err = np.abs(x.reshape(-1, 32).astype(np.float64) - df[:, None] * q.reshape(-1, 32))
    assert np.all(err <= df[:, None] * (0.5 + 1e-5))
    assert q.min() >= -127 and q.max() <= 127
    assert np.all(np.abs(q.reshape(-1, 32)).max(axis=1) == 127)


def test_q8_0_lanes_brute_force_and_unit_scale_exact():
    rng = np.random.default_rng(11)
    R, K = 9, 128
    qs = rng.integers(-127, 128, size=(R, K)).astype(np.int8)
    one = np.full((R, K // 32), 0x3C00, dtype=np.uint16)   # fp16 1.0
    x = rng.integers(-50, 51, size=K).astype(np.float64)
    y = oracle.gemv_q8_0(qs, one, x=x, act="f32")
    assert list(y.astype(np.int64)) == [sum(int(qs[r, c]) * int(x[c]) for c in range(K)) for r in range(R)]
    # dp4a lane against a pure-Python evaluation of its definition
    d = (np.abs(rng.standard_normal((R, K // 32))) * 0.002).astype(np.float16).view(np.uint16)
    xf = rng.standard_normal(K).astype(np.float32)
    xq, xd = oracle.q8_0_quantize(xf)
    y = oracle.gemv_q8_0(qs, d, xq=xq, xd_bits=xd, act="i8")
    for r in range(R):
        tot = 0.0
        for b in range(K // 32):
            dot = sum(int(qs[r, 32 * b + i]) * int(xq[32 * b + i]) for i in range(32))
            tot += float(np.float16(d[r, b].view(np.float16))) * float(xd[b].view(np.float16)) * dot
        assert y[r] == pytest.approx(tot, rel=1e-12, abs=1e-12)
    dots = oracle.q8_0_block_dots(qs, xq)
    assert dots[2, 1] == sum(int(qs[2, 32 + i]) * int(xq[32 + i]) for i in range(32))


def _golden_widen():
    rows = []
    with open(os.path.join(GOLDEN, "q8_0_widen_bf16_hand.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                q, d, w = line.split()
                rows.append((int(q), int(d, 16), int(w, 16)))
    return rows


@pytest.mark.parametrize("q,d,w", _golden_widen())
def test_q8_0_widen_bf16_hand_cases(q, d, w):
    got = oracle.f64_to_bf16_bits(oracle.q8_0_widen_bf16(np.full((1, 32), q, dtype=np.int8),
                                                         np.array([[d]], dtype=np.uint16)))
    assert np.all(got == w), (hex(int(got[0, 0])), hex(w))


def _bf16_rne_exact(v):
    """Round a Fraction to 8 significant bits, ties to even, in exact rational arithmetic."""
    from fractions import Fraction
    if v == 0:
        return Fraction(0)
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    scale = Fraction(2) ** (7 - e)          # a * scale lies in [128, 256)
    m = a * scale
    lo = m.numerator // m.denominator
    rem = m - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return (lo / scale) * (1 if v > 0 else -1)


def test_q8_0_widened_lane_brute_force_and_power_of_two_scales():
    from fractions import Fraction
    rng = np.random.default_rng(12)
    R, K = 5, 96
    qs = rng.integers(-128, 128, size=(R, K)).astype(np.int8)
    d = (np.abs(rng.standard_normal((R, K // 32))) * 0.01).astype(np.float16).view(np.uint16)
    x = rng.integers(-8, 9, size=K).astype(np.float64)
    y = oracle.gemv_q8_0(qs, d, x=x, act="w_bf16")
    rounded = 0
    for r in range(R):
        tot = Fraction(0)
        for k in range(K):
            exact = Fraction(float(d[r, k // 32].view(np.float16))) * int(qs[r, k])
            w = _bf16_rne_exact(exact)
            rounded += w != exact
            tot += w * int(x[k])
        assert y[r] == pytest.approx(float(tot), rel=1e-13, abs=1e-13)
    assert rounded > R * K // 2        # the random scales do make most weights round
    # power-of-two scales: widening is exact, so the lane equals the dequantising lane
    p2 = np.array([0x3C00, 0x3800, 0x4000], dtype=np.uint16)[rng.integers(0, 3, (R, K // 32))]
    np.testing.assert_array_equal(oracle.gemv_q8_0(qs, p2, x=x, act="w_bf16"),
                                  oracle.gemv_q8_0(qs, p2, x=x, act="f32"))


def test_q8_0_dequant_layout():
    qs = np.arange(-32, 32, dtype=np.int8).reshape(1, 64)
    d = np.array([[0x3C00, 0x4000]], dtype=np.uint16)      # 1.0, 2.0
    w = oracle.q8_0_dequant(qs, d)
    np.testing.assert_array_equal(w[0, :32], np.arange(-32, 0))
    np.testing.assert_array_equal(w[0, 32:], 2 * np.arange(0, 32))


# ---------------------------------------------------------------- argmax, paging


def test_argmax_rules():
    assert oracle.argmax_first([1.0, 3.0, 3.0, 2.0]) == 1
    assert oracle.argmax_first([np.nan, 1.0, 0.5]) == 1
    assert oracle.argmax_first([0.0, 1.0, np.nan, 5.0]) == 3
    assert oracle.argmax_first([-np.inf, -np.inf]) == 0
    assert oracle.argmax_first([np.nan, np.nan]) == 0
    x = np.zeros(151936)
    x[-1] = 1e-30
    assert oracle.argmax_first(x) == 151935


def test_paged_indices_and_gather():
    pt = np.array([3, 0, 2, 1])
    assert [oracle.paged_token_index(pt, t, 4) for t in (0, 3, 4, 9, 15)] == [12, 15, 0, 9, 7]
    rng = np.random.default_rng(12)
    logical = rng.standard_normal((2, 16, 8))
    pages = np.zeros((4, 2, 4, 8))
    for t in range(16):
        pages[pt[t // 4], :, t % 4, :] = logical[:, t, :]
    np.testing.assert_array_equal(oracle.gather_paged(pages, pt, 16), logical)


# ---------------------------------------------------------------- one layer


def _tiny_layer(rng, H=256, hq=4, hkv=2, D=128, F=96, zero_out=False):
    b = lambda a: oracle.f64_to_bf16_bits(a)  # noqa: E731
    lw = oracle.LayerWeights(
        w_qkv=b(rng.standard_normal(((hq + 2 * hkv) * D, H)) * 0.02),
        w_o=b(np.zeros((H, hq * D)) if zero_out else rng.standard_normal((H, hq * D)) * 0.02),
        w_gu=b(rng.standard_normal((2 * F, H)) * 0.02),
        w_down=b(np.zeros((H, F)) if zero_out else rng.standard_normal((H, F)) * 0.02),
        ln_in=b(1 + 0.1 * rng.standard_normal(H)), ln_post=b(1 + 0.1 * rng.standard_normal(H)),
        q_norm=b(1 + 0.1 * rng.standard_normal(D)), k_norm=b(1 + 0.1 * rng.standard_normal(D)))
    return oracle.Dims(H, hq, hkv, D, F), lw


def test_layer_zero_outputs_leave_residual_and_write_cache():
    rng = np.random.default_rng(13)
    dims, lw = _tiny_layer(rng, zero_out=True)
    res = rng.standard_normal(256)
    kc, vc = np.zeros((2, 10, 128)), np.zeros((2, 10, 128))
    out = oracle.layer_step(dims, lw, res, kc, vc, pos=4, mode="exact", act="bf16")
    np.testing.assert_array_equal(out, res)
    assert np.count_nonzero(kc[:, 4]) > 0 and np.count_nonzero(vc[:, 4]) > 0
    assert np.count_nonzero(kc[:, 5:]) == 0 and np.count_nonzero(kc[:, :4]) == 0


def test_layer_first_token_attention_is_its_value():
    # pos = 0: a single visible key, so each q head's output is v of its kv head;
    # the layer's first residual update is then W_o applied to the repeated v.
    rng = np.random.default_rng(14)
    dims, lw = _tiny_layer(rng)
    res = rng.standard_normal(256)
    kc, vc = np.zeros((2, 1, 128)), np.zeros((2, 1, 128))
    tr = {}
    oracle.layer_step(dims, lw, res, kc, vc, pos=0, mode="exact", act="bf16", trace=tr)
    qkv = oracle.bf16_to_f64(lw.w_qkv) @ tr["xn"]
    v = qkv[6 * 128:].reshape(2, 128)
    np.testing.assert_allclose(tr["attn"].reshape(4, 128), v[[0, 0, 1, 1]], rtol=1e-12)
    # k in the cache has the RMS of the k_norm-weighted unit vector, rotated (pos 0 = identity)
    kn = qkv[4 * 128:6 * 128].reshape(2, 128)
    for g in range(2):
        rms = math.sqrt(float(np.mean(kn[g] ** 2)) + 1e-6)
        np.testing.assert_allclose(kc[g, 0], oracle.bf16_to_f64(lw.k_norm) * kn[g] / rms, rtol=1e-12)


def test_decode_token_structure():
    # two layers with zero output projections: final residual is the embedding row,
    # so logits are the (tied) LM head applied to the final RMSNorm of that row.
    rng = np.random.default_rng(15)
    dims, l0 = _tiny_layer(rng, zero_out=True)
    _, l1 = _tiny_layer(rng, zero_out=True)
    V = 300
    emb = oracle.f64_to_bf16_bits(rng.standard_normal((V, 256)) * 0.02)
    fn = oracle.f64_to_bf16_bits(1 + 0.1 * rng.standard_normal(256))
    m = oracle.Model(dims, [l0, l1], emb, fn, emb)
    ks = [np.zeros((2, 8, 128)) for _ in range(2)]
    vs = [np.zeros((2, 8, 128)) for _ in range(2)]
    logits = oracle.decode_token(m, 17, 3, ks, vs, mode="exact")
    e = oracle.bf16_to_f64(emb)
    xf = e[17] / math.sqrt(float(np.mean(e[17] ** 2)) + 1e-6) * oracle.bf16_to_f64(fn)
    np.testing.assert_allclose(logits, e @ xf, rtol=1e-10, atol=1e-14)
