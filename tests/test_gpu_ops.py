"""Parity of each C-ABI kernel with the CPU oracle, element by element.

Sizes span several CTAs and ragged tails; the full-size shapes of the decode
workloads (Qwen3-0.6B / Qwen3-8B projections, the 151936-row LM head) are run
too. Floating-point outputs are compared with a relative max-abs error
(max |gpu - ref| / max |ref|); integer and index outputs bit-exactly.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from transformer_decode_step_weight_gb300 import api, synth
from helpers import rel_max_abs

pytestmark = pytest.mark.gpu
DEV = "cuda"
# f32 accumulation of bf16 products over K <= 12288 terms vs float64
GEMV_TOL = 2e-5


def _gen(seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return g


@pytest.mark.parametrize("R,K,B", [(1, 8, 1), (37, 96, 1), (333, 136, 1), (1000, 1024, 1), (4096, 2048, 1),
                                   (6144, 4096, 1), (4096, 12288, 1), (2000, 3072, 2), (513, 4096, 3),
                                   (1024, 4096, 8), (300, 20000, 1), (151936, 1024, 1)])
def test_gemv_bf16(cuda_lib, R, K, B):
    g = _gen(R + K)
    W = (torch.randn((R, K), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    x = torch.randn((B, K), generator=g, device=DEV).to(torch.bfloat16)
    y = api.gemv_bf16(W, x)
    torch.cuda.synchronize()
    Wb, xb = synth.bits_u16(W), synth.bits_u16(x)
    for b in range(B):
        ref = oracle.gemv_bf16(Wb, oracle.bf16_to_f64(xb[b]))
        assert rel_max_abs(y[b].cpu().numpy(), ref) < GEMV_TOL


# batch 2..8, bf16 x: the mma.sync weight-streaming GEMV (QD_SMALLB_IMPL=simt: the
# CUDA-core GEMV). Rows below the SM count, ragged 32-row stages, K in one 32-column
# chunk, past the 4096 columns held in registers with a ragged last stage, and the
# Qwen3-8B / 0.6B projection and LM-head shapes.
@pytest.mark.parametrize("R,K,B", [(1, 32, 2), (37, 96, 2), (151, 4128, 5), (153, 544, 8), (2000, 3072, 2),
                                   (513, 4096, 3), (1024, 4096, 8), (4096, 12288, 8), (3000, 8224, 7),
                                   (24576, 4096, 4), (151936, 1024, 4), (151936, 4096, 8)])
@pytest.mark.parametrize("impl", ["mma", "simt"])
def test_gemv_bf16_small_batch(cuda_lib, monkeypatch, impl, R, K, B):
    monkeypatch.setenv("QD_SMALLB_IMPL", impl)
    g = _gen(R * 3 + K + B)
    W = (torch.randn((R, K), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    x = torch.randn((B, K), generator=g, device=DEV).to(torch.bfloat16)
    try:
        y = api.gemv_bf16(W, x)
    except api.QDError:
        if impl == "mma":
            raise
        pytest.skip("the CUDA-core GEMV takes this K only at a smaller batch")
    torch.cuda.synchronize()
    Wb, xb = synth.bits_u16(W), synth.bits_u16(x)
    rows = np.arange(R) if R <= 8192 else np.arange(0, R, 53)
    for b in range(B):
        ref = oracle.gemv_bf16(Wb[rows], oracle.bf16_to_f64(xb[b]))
        assert rel_max_abs(y[b].cpu().numpy()[rows], ref) < GEMV_TOL, b


def test_gemv_bf16_small_batch_integer_exact(cuda_lib):
    # small integers: every product and partial sum exact in binary32, so the mma.sync
    # GEMV must give the exact integer result at every batch 2..8
    g = _gen(29)
    W = torch.randint(-8, 9, (333, 4160), generator=g, device=DEV).to(torch.bfloat16)
    for B in range(2, 9):
        x = torch.randint(-8, 9, (B, 4160), generator=g, device=DEV).to(torch.bfloat16)
        y = api.gemv_bf16(W, x)
        ref = x.double().cpu() @ W.double().cpu().T
        assert torch.equal(y.cpu().double(), ref), B


@pytest.mark.parametrize("R,K,B", [(128, 64, 9), (300, 1024, 16), (4096, 4096, 64), (1000, 12288, 33),
                                   (6144, 4096, 64), (151936, 4096, 64), (300, 1024, 65), (1000, 4096, 200),
                                   (4096, 4096, 512)])
def test_gemm_bf16_tensor_cores(cuda_lib, R, K, B):
    # batch >= 9: the tcgen05 path (ragged last 128-row tile, batch below 64; above 64
    # the prompt-row form, 64-row tiles of x over the grid with a ragged last one)
    g = _gen(R * 7 + B)
    W = (torch.randn((R, K), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    x = torch.randn((B, K), generator=g, device=DEV).to(torch.bfloat16)
    y = api.gemv_bf16(W, x)
    torch.cuda.synchronize()
    Wb, xb = synth.bits_u16(W), synth.bits_u16(x)
    rows = np.arange(R) if R <= 8192 else np.arange(0, R, 97)
    for b in sorted({0, B // 2, B - 1}):
        ref = oracle.gemv_bf16(Wb[rows], oracle.bf16_to_f64(xb[b]))
        assert rel_max_abs(y[b].cpu().numpy()[rows], ref) < GEMV_TOL, b


# many token rows (prefill): the persistent form (one CTA per SM over (weight tile,
# 256-token tile) items, two TMEM accumulators, the default) and the one-CTA-per-tile
# form (QD_GEMM_WIDE=tiles); ragged weight and token tiles, and more items than CTAs.
# The residual-add epilogue runs in the prefill tests (O and down projections).
@pytest.mark.parametrize("R,K,B", [(300, 1024, 300), (1000, 4096, 200), (4096, 4096, 512), (6144, 4096, 2048),
                                   (24576, 4096, 1030)])
@pytest.mark.parametrize("form", ["persistent", "tiles"])
def test_gemm_bf16_wide(cuda_lib, monkeypatch, R, K, B, form):
    monkeypatch.setenv("QD_GEMM_WIDE", form)
    g = _gen(R + B + K)
    W = (torch.randn((R, K), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    x = torch.randn((B, K), generator=g, device=DEV).to(torch.bfloat16)
    y = api.gemv_bf16(W, x)
    torch.cuda.synchronize()
    Wb, xb = synth.bits_u16(W), synth.bits_u16(x)
    rows = np.arange(R) if R <= 8192 else np.arange(0, R, 97)
    for b in sorted({0, B // 3, B - 1}):
        ref = oracle.gemv_bf16(Wb[rows], oracle.bf16_to_f64(xb[b]))
        assert rel_max_abs(y[b].cpu().numpy()[rows], ref) < GEMV_TOL, b


def test_gemm_bf16_tensor_cores_integer_exact(cuda_lib):
    g = _gen(13)
    W = torch.randint(-8, 9, (384, 512), generator=g, device=DEV).to(torch.bfloat16)
    for B in (24, 130):
        x = torch.randint(-8, 9, (B, 512), generator=g, device=DEV).to(torch.bfloat16)
        y = api.gemv_bf16(W, x)
        ref = x.double().cpu() @ W.double().cpu().T
        assert torch.equal(y.cpu().double(), ref), B


def test_gemv_bf16_f32_input_rounds_to_bf16(cuda_lib):
    g = _gen(5)
    W = (torch.randn((700, 4096), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    x = torch.randn((1, 4096), generator=g, device=DEV)
    y = api.gemv_bf16(W, x)
    ref = oracle.gemv_bf16(synth.bits_u16(W), oracle.round_bf16(x[0].cpu().numpy()))
    assert rel_max_abs(y[0].cpu().numpy(), ref) < GEMV_TOL


def test_gemv_bf16_integer_exact(cuda_lib):
    # integer-valued bf16 W and x with |partial sums| < 2^24: exact in any order
    g = _gen(6)
    W = torch.randint(-8, 9, (513, 1024), generator=g, device=DEV).to(torch.bfloat16)
    x = torch.randint(-8, 9, (1, 1024), generator=g, device=DEV).to(torch.bfloat16)
    y = api.gemv_bf16(W, x)
    ref = W.double().cpu() @ x[0].double().cpu()
    assert torch.equal(y[0].cpu().double(), ref)


def _q8(R, K, seed):
    g = _gen(seed)
    qs = torch.randint(-127, 128, (R, K), generator=g, device=DEV, dtype=torch.int16).to(torch.int8)
    d = (torch.randn((R, K // 32), generator=g, device=DEV).abs() * 0.002).to(torch.float16)
    return qs, d


def test_quantize_q8_0_bit_exact(cuda_lib):
    g = _gen(7)
    x = torch.randn(12288, generator=g, device=DEV) * 3
    x[64:96] = 0.0                      # d = 0 block
    x[96:128] = torch.linspace(-127, 127, 32, device=DEV)
    xq, xd = api.quantize_q8_0(x)
    rq, rd = oracle.q8_0_quantize(x.cpu().numpy())
    assert np.array_equal(xq.cpu().numpy(), rq)
    assert np.array_equal(synth.bits_u16(xd), rd)


@pytest.mark.parametrize("R,K", [(33, 64), (513, 96), (1000, 1024), (4096, 4096), (3000, 12288), (6144, 4096)])
def test_q8_block_dots_bit_exact(cuda_lib, R, K):
    # the production i8-lane GEMV stores the int32 block dots it forms (K % 256 == 0:
    # the TMA-ring form the decode step runs; otherwise the register-streaming form)
    qs, d = _q8(R, K, R)
    x = torch.randn(K, generator=_gen(K), device=DEV)
    xq, xd = api.quantize_q8_0(x)
    dots, y = api.debug_q8_block_dots(qs, d, xq, xd)
    torch.cuda.synchronize()
    ref = oracle.q8_0_block_dots(synth.host_i8(qs), synth.host_i8(xq))
    assert np.array_equal(dots.cpu().numpy().astype(np.int64), ref)
    yref = oracle.gemv_q8_0(synth.host_i8(qs), synth.bits_u16(d), xq=synth.host_i8(xq), xd_bits=synth.bits_u16(xd),
                            act="i8")
    assert rel_max_abs(y.cpu().numpy(), yref) < GEMV_TOL
    # the same launch without the dump gives the same bits
    y2 = api.gemv_q8_0(qs, d, xq=xq, xd=xd, act=api.QD_ACT_I8)
    assert torch.equal(y, y2)


@pytest.mark.parametrize("R,K", [(37, 64), (1000, 1024), (6144, 4096), (4096, 12288), (151936, 1024)])
def test_gemv_q8_0_f32_lane(cuda_lib, R, K):
    qs, d = _q8(R, K, R + 1)
    x = torch.randn(K, generator=_gen(K + 1), device=DEV)
    y = api.gemv_q8_0(qs, d, x=x, act=api.QD_ACT_F32)
    ref = oracle.gemv_q8_0(synth.host_i8(qs), synth.bits_u16(d), x=x.cpu().numpy().astype(np.float64), act="f32")
    assert rel_max_abs(y.cpu().numpy(), ref) < GEMV_TOL


@pytest.mark.parametrize("R,K", [(37, 64), (1000, 1024), (6144, 4096), (4096, 12288)])
def test_gemv_q8_0_i8_lane(cuda_lib, R, K):
    qs, d = _q8(R, K, R + 2)
    x = torch.randn(K, generator=_gen(K + 2), device=DEV)
    xq, xd = api.quantize_q8_0(x)
    y = api.gemv_q8_0(qs, d, xq=xq, xd=xd, act=api.QD_ACT_I8)
    ref = oracle.gemv_q8_0(synth.host_i8(qs), synth.bits_u16(d), xq=synth.host_i8(xq), xd_bits=synth.bits_u16(xd),
                           act="i8")
    assert rel_max_abs(y.cpu().numpy(), ref) < GEMV_TOL
    # the lane that quantises in its own prologue gives the same codes, so the same result
    y2 = api.gemv_q8_0(qs, d, x=x, act=api.QD_ACT_I8)
    assert rel_max_abs(y2.cpu().numpy(), ref) < GEMV_TOL


def test_gemv_q8_0_unit_scales_integer_exact(cuda_lib):
    qs, _ = _q8(700, 1024, 9)
    d = torch.ones((700, 32), dtype=torch.float16, device=DEV)
    x = torch.randint(-40, 41, (1024,), generator=_gen(10), device=DEV).float()
    y = api.gemv_q8_0(qs, d, x=x, act=api.QD_ACT_F32)
    ref = qs.double().cpu() @ x.double().cpu()
    assert torch.equal(y.cpu().double(), ref)


@pytest.mark.parametrize("R,K,B,split", [(128, 256, 2, False), (300, 768, 17, False), (1000, 1536, 64, True),
                                         (6144, 4096, 64, True), (4096, 12288, 64, True),
                                         (151936, 4096, 64, False), (300, 768, 130, False)])
def test_gemm_q8_0_tensor_cores(cuda_lib, R, K, B, split, parity_log):
    # Q8_0 weights widened to bf16 on chip: ragged last 128-row tile, batch below 64,
    # K split across CTAs (partials summed in split order) where the grid is small.
    # Held to the widened-weight lane element by element and to the pages' Q8_0
    # definition w = f32(d) q at the bf16 path's tolerance (the widening error).
    qs, d = _q8(R, K, R + 5)
    x = torch.randn((B, K), generator=_gen(K + 5), device=DEV).to(torch.bfloat16)
    ws = None
    if split:
        nbytes = api.gemm_workspace_bytes(R, K)
        assert nbytes > 0
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    y = api.gemm_q8_0(qs, d, x, workspace=ws)
    y2 = api.gemm_q8_0(qs, d, x, workspace=ws)   # the first call left its tickets at zero
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    qh, dh, xb = synth.host_i8(qs), synth.bits_u16(d), synth.bits_u16(x)
    rows = np.arange(R) if R <= 8192 else np.arange(0, R, 97)
    worst = 0.0
    for b in sorted({0, B // 2, B - 1}):
        ref = oracle.gemv_q8_0(qh[rows], dh[rows], x=oracle.bf16_to_f64(xb[b]), act="w_bf16")
        assert rel_max_abs(y[b].cpu().numpy()[rows], ref) < GEMV_TOL, b
        ref = oracle.gemv_q8_0(qh[rows], dh[rows], x=oracle.bf16_to_f64(xb[b]), act="f32")
        err = rel_max_abs(y[b].cpu().numpy()[rows], ref)
        worst = max(worst, err)
        assert err < 2e-2, (b, err)
    parity_log[f"gemm_q8_0_vs_q8_0_definition/{R}x{K}x{B}"] = worst
    assert api.check_device_error() == 0


def test_gemm_q8_0_widening_bit_exact(cuda_lib):
    # one-hot activations pick single widened weights, y[b, r] = bf16(f32(d[r, c_b / 32]) * q[r, c_b])
    # exactly: this pins the swizzled placement and the scale of each column position
    R, K, B = 200, 256, 64
    qs, d = _q8(R, K, 77)
    cols = np.arange(B) * 4 + np.arange(B) // 16       # all four K tiles, every 16-byte chunk
    x = torch.zeros((B, K), dtype=torch.bfloat16, device=DEV)
    x[torch.arange(B, device=DEV), torch.tensor(cols, device=DEV)] = 1.0
    y = api.gemm_q8_0(qs, d, x)
    W = oracle.q8_0_widen_bf16(synth.host_i8(qs), synth.bits_u16(d))
    np.testing.assert_array_equal(y.cpu().numpy().astype(np.float64), W[:, cols].T)


def test_gemm_q8_0_unit_scales_integer_exact(cuda_lib):
    qs, _ = _q8(384, 512, 21)
    d = torch.ones((384, 16), dtype=torch.float16, device=DEV)
    x = torch.randint(-8, 9, (24, 512), generator=_gen(22), device=DEV).to(torch.bfloat16)
    y = api.gemm_q8_0(qs, d, x)
    ref = x.double().cpu() @ qs.double().cpu().T
    assert torch.equal(y.cpu().double(), ref)


# ---------------------------------------------------------------- attention


def _attn_case(B, hq, hkv, lens, ps, seed, paged=True):
    g = _gen(seed)
    D = 128
    if paged:
        per = [max(1, -(-n // ps)) for n in lens]
        max_pages = max(per)
        n_pages = sum(per) + 3
        perm = torch.randperm(n_pages, generator=g, device=DEV).to(torch.int32)
        pt = torch.zeros((B, max_pages), dtype=torch.int32, device=DEV)
        off = 0
        for b, n in enumerate(per):
            pt[b, :n] = perm[off:off + n]
            off += n
    else:
        ps = max(lens) + 5
        max_pages, n_pages = 1, B
        pt = torch.arange(B, dtype=torch.int32, device=DEV).reshape(B, 1)
    kp = torch.randn((n_pages, hkv, ps, D), generator=g, device=DEV).to(torch.bfloat16)
    vp = torch.randn((n_pages, hkv, ps, D), generator=g, device=DEV).to(torch.bfloat16)
    q = torch.randn((B, hq, D), generator=g, device=DEV) * 0.3
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    return q, kp, vp, pt, sl


def _attn_ref(q, kp, vp, pt, lens):
    out = []
    for b, n in enumerate(lens):
        if n == 0:
            out.append(np.zeros((q.shape[1], 128)))
            continue
        k = oracle.bf16_to_f64(oracle.gather_paged(synth.bits_u16(kp), pt[b].cpu().numpy(), n))
        v = oracle.bf16_to_f64(oracle.gather_paged(synth.bits_u16(vp), pt[b].cpu().numpy(), n))
        out.append(oracle.gqa_attention(q[b].double().cpu().numpy(), k, v))
    return np.stack(out)


@pytest.mark.parametrize("B,hq,hkv,lens,ps,paged", [
    (1, 4, 2, [1], 16, False), (1, 4, 2, [64], 16, False), (1, 4, 2, [65], 16, False),
    (1, 16, 8, [129], 16, False), (1, 32, 8, [4224], 16, False), (2, 8, 8, [5, 1000], 16, False),
    (3, 32, 8, [1, 37, 300], 16, True), (4, 16, 2, [17, 64, 128, 700], 16, True),
    (2, 8, 1, [100, 33], 7, True), (5, 4, 4, [0, 3, 64, 65, 2000], 32, True),
    # 32 .. SM-count (sequence, kv head) pairs: the tensor-core form with the CUDA-core
    # form's split sizing (TMA boxes at 16-token pages, cp.async at 8)
    (6, 32, 8, [1, 64, 65, 700, 1500, 3000], 16, True), (4, 16, 8, [3, 129, 640, 2049], 8, True)])
def test_attention_parity(cuda_lib, B, hq, hkv, lens, ps, paged):
    q, kp, vp, pt, sl = _attn_case(B, hq, hkv, lens, ps, B * 100 + hq + sum(lens), paged)
    out = api.attn_decode_paged(q, kp, vp, pt, sl, 1 / math.sqrt(128))
    ref = _attn_ref(q, kp, vp, pt, lens)
    got = out.cpu().numpy()
    for b, n in enumerate(lens):
        if n == 0:
            assert np.all(got[b] == 0)
        else:
            assert rel_max_abs(got[b], ref[b]) < 1e-5, (b, n)
    assert api.check_device_error() == 0


@pytest.mark.parametrize("ps,with_empty", [(16, False), (32, True), (8, False)])
def test_attention_parity_tensor_core_form(cuda_lib, ps, with_empty):
    """20 sequences x 8 kv heads (at least one CTA per SM) take the tensor-core form:
    1024-token splits, K/V by 2D TMA when the page size is a multiple of 16 (16, 32),
    by 16-byte cp.async otherwise (8). Lengths cross split, tile and page edges."""
    g = torch.Generator().manual_seed(ps)
    lens = [int(v) for v in torch.randint(1, 2600, (20,), generator=g)]
    lens[3], lens[7], lens[11] = 1024, 1025, 63
    if with_empty:
        lens[5] = 0
    q, kp, vp, pt, sl = _attn_case(20, 32, 8, lens, ps, 900 + ps, True)
    out = api.attn_decode_paged(q, kp, vp, pt, sl, 1 / math.sqrt(128))
    ref = _attn_ref(q, kp, vp, pt, lens)
    got = out.cpu().numpy()
    for b, n in enumerate(lens):
        if n == 0:
            assert np.all(got[b] == 0)
        else:
            assert rel_max_abs(got[b], ref[b]) < 1e-5, (b, n)
    assert api.check_device_error() == 0


def test_attention_page_permutation_is_bitwise_invariant(cuda_lib):
    # same logical cache through a permuted page table == identity table over permuted data
    lens = [300, 77]
    q, kp, vp, pt, sl = _attn_case(2, 32, 8, lens, 16, 42, True)
    out1 = api.attn_decode_paged(q, kp, vp, pt, sl, 1 / math.sqrt(128))
    # lay each sequence's used pages out in logical order and point an identity-like table at them
    new_pt = torch.zeros_like(pt)
    kp2, vp2 = torch.zeros_like(kp), torch.zeros_like(vp)
    nxt = 0
    for b, n in enumerate(lens):
        for j in range(-(-n // 16)):
            src = int(pt[b, j])
            kp2[nxt], vp2[nxt] = kp[src], vp[src]
            new_pt[b, j] = nxt
            nxt += 1
    out2 = api.attn_decode_paged(q, kp2, vp2, new_pt, sl, 1 / math.sqrt(128))
    assert torch.equal(out1, out2)


def test_attention_is_deterministic(cuda_lib):
    q, kp, vp, pt, sl = _attn_case(2, 32, 8, [4000, 2500], 16, 7, True)
    ws = torch.zeros(api.attn_workspace_bytes(2, 32, 8, pt.shape[1] * 16), dtype=torch.uint8, device=DEV)
    a = api.attn_decode_paged(q, kp, vp, pt, sl, 0.088, workspace=ws)
    b = api.attn_decode_paged(q, kp, vp, pt, sl, 0.088, workspace=ws)
    assert torch.equal(a, b)
    assert torch.count_nonzero(ws[-256:]) == 0   # tickets (last 256-byte block) reset to zero


def test_paged_indices_bit_exact(cuda_lib):
    # through the page-table lookup the attention kernels use
    g = _gen(11)
    pt = torch.randperm(40, generator=g, device=DEV).to(torch.int32).reshape(4, 10)
    idx = api.debug_paged_indices(pt, 16, 150, n_pages=40)
    ptn = pt.cpu().numpy()
    ref = np.array([[oracle.paged_token_index(ptn[b], t, 16) for t in range(150)] for b in range(4)])
    assert np.array_equal(idx.cpu().numpy(), ref)
    for ps in (1, 7, 32):
        idx = api.debug_paged_indices(pt, ps, 10 * ps, n_pages=40)
        ref = np.array([[oracle.paged_token_index(ptn[b], t, ps) for t in range(10 * ps)] for b in range(4)])
        assert np.array_equal(idx.cpu().numpy(), ref), ps
    assert api.check_device_error() == 0
    # an id outside the cache is not followed: -1 there and the page error bit
    pt[1, 2] = 40
    idx = api.debug_paged_indices(pt, 16, 150, n_pages=40).cpu().numpy()
    assert np.all(idx[1, 32:48] == -1) and np.all(idx[1, :32] >= 0) and np.all(idx[1, 48:] >= 0)
    assert api.check_device_error() == 1


def test_rope_table_matches_definition(cuda_lib):
    t = api.rope_table(4224, 128, 1e6, DEV).cpu().numpy().astype(np.float64)
    for pos in (0, 1, 127, 4223):
        e = np.zeros(128)
        e[:64] = 1.0
        r = oracle.rope(e, pos)                  # (cos a_i, sin a_i) for a unit first half
        np.testing.assert_allclose(t[pos, :, 0], r[:64], atol=2e-7)
        np.testing.assert_allclose(t[pos, :, 1], r[64:], atol=2e-7)


# ---------------------------------------------------------------- argmax


def test_argmax_advance_rules(cuda_lib):
    V = 151936
    lg = torch.randn((6, V), generator=_gen(12), device=DEV)
    lg[0, 77] = 50.0
    lg[0, 78] = 50.0                    # tie -> lowest index
    lg[1, V - 1] = 1e9                  # maximum at the last index
    lg[2, :] = float("nan")
    lg[2, 5] = 1.0                      # NaN never wins
    lg[3, :] = -float("inf")            # all -inf -> index 0
    lg[4, 1000:] = float("nan")
    tok = torch.zeros(6, dtype=torch.int32, device=DEV)
    pos = torch.arange(6, dtype=torch.int32, device=DEV) * 10
    step = torch.zeros(6, dtype=torch.int32, device=DEV)
    out = torch.full((6, 4), -1, dtype=torch.int32, device=DEV)
    api.argmax_advance(lg, tok, pos, step, out)
    exp = [oracle.argmax_first(r) for r in lg.cpu().numpy()]
    assert tok.tolist() == exp
    assert exp[:4] == [77, V - 1, 5, 0]
    assert out[:, 0].tolist() == exp and pos.tolist() == [1, 11, 21, 31, 41, 51] and step.tolist() == [1] * 6
    assert api.check_device_error() == 0
    lg[5, :] = float("nan")             # all-NaN row: token 0 and the NaN error bit
    step.fill_(4)                       # out_tokens full: STEPS error bit, no write
    api.argmax_advance(lg, tok, pos, step, out)
    assert tok[5].item() == 0
    assert api.check_device_error() == (4 | 8)
    assert api.check_device_error() == 0


def test_bounded_wait_times_out_and_the_context_stays_usable(cuda_lib):
    # a wait on an mbarrier that no copy completes gives up after its limit, sets the
    # timeout bit and returns; the next kernel runs normally
    import time
    assert api.check_device_error() == 0
    t0 = time.perf_counter()
    api.debug_wait_timeout(2000)
    bits = api.check_device_error()
    dt = time.perf_counter() - t0
    assert bits == 16, bits            # QD_DEVERR_TIMEOUT alone
    assert dt < 5.0
    g = _gen(99)
    W = (torch.randn((300, 512), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    x = torch.randn((1, 512), generator=g, device=DEV).to(torch.bfloat16)
    y = api.gemv_bf16(W, x)
    ref = oracle.gemv_bf16(synth.bits_u16(W), oracle.bf16_to_f64(synth.bits_u16(x[0])))
    assert rel_max_abs(y[0].cpu().numpy(), ref) < GEMV_TOL
    assert api.check_device_error() == 0
