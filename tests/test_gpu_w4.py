"""W4A16 (INT4 weights, bf16 activations): the GEMV, the INT4 LM head with its local
top-k, and the whole step, against the oracle.

"GPU Kernel Lab" README, "Quantization experiments": W4A16 decode GEMV and packed INT4
LM head with local top-k, per-output-channel weight quantization.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL, oracle_caches, oracle_model, rel_max_abs, teacher_forced
from transformer_decode_step_weight_gb300 import api, synth

pytestmark = pytest.mark.gpu
DEV = "cuda"
GEMV_TOL = 2e-5


@pytest.fixture(params=["mma", "tc"], autouse=True)
def w4_impl(request, monkeypatch):
    """Every test runs on both INT4 forms: mma.sync (the default) and tcgen05 (K a
    multiple of 256; the library reads QD_W4_IMPL on every call)."""
    monkeypatch.setenv("QD_W4_IMPL", request.param)
    return request.param


def _w4(R, K, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    q = torch.randint(0, 16, (R, K), generator=g, device=DEV, dtype=torch.int16)
    W = (q[:, 0::2] | (q[:, 1::2] << 4)).to(torch.uint8)
    d = (torch.randn(R, generator=g, device=DEV).abs() * 0.01).to(torch.float16)
    x = torch.randn(K, generator=g, device=DEV).to(torch.bfloat16)
    return W, d, x


@pytest.mark.parametrize("R,K", [(37, 64), (1000, 1024), (333, 2048), (300, 2080), (4096, 3072), (6144, 4096),
                                 (4096, 12288), (77, 16384), (151936, 1024)])
def test_gemv_w4(cuda_lib, R, K):
    W, d, x = _w4(R, K, R + K)
    y = api.gemv_w4(W, d, x)
    ref = oracle.gemv_w4(synth.host_u8(W), synth.bits_u16(d), oracle.bf16_to_f64(synth.bits_u16(x)))
    assert rel_max_abs(y.cpu().numpy(), ref) < GEMV_TOL


@pytest.mark.parametrize("R,K", [(37, 1024), (4096, 4096), (6144, 4096), (4096, 12288), (300, 16384),
                                 (1000, 256)])
def test_gemv_w4_split_k(cuda_lib, R, K):
    # the tcgen05 form with a workspace: tiles that underfill the SMs split K, the last
    # split adds the partials in split order; two calls (the tickets are left at zero)
    W, d, x = _w4(R, K, 3 * R + K)
    nbytes = api.gemv_w4_workspace_bytes(R, K)
    ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=DEV)
    y1 = api.gemv_w4(W, d, x, workspace=ws)
    y2 = api.gemv_w4(W, d, x, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    ref = oracle.gemv_w4(synth.host_u8(W), synth.bits_u16(d), oracle.bf16_to_f64(synth.bits_u16(x)))
    assert rel_max_abs(y1.cpu().numpy(), ref) < GEMV_TOL
    assert api.check_device_error() == 0


def test_gemv_w4_rejects_unsupported_k(cuda_lib):
    for K in (48, 16416):   # not a multiple of 32; above the 16384-column maximum
        W, d, x = _w4(16, K, 1)
        with pytest.raises(api.QDError):
            api.gemv_w4(W, d, x)


def test_gemv_w4_unit_scales_integer_exact(cuda_lib):
    # small integer activations: every partial sum of (1 + u/16) x is a multiple of 1/16
    # below 2^20, so the f32 result is the exact integer sum q x
    W, _, _ = _w4(700, 1024, 5)
    d = torch.ones(700, dtype=torch.float16, device=DEV)
    x = torch.randint(-8, 9, (1024,), generator=torch.Generator(device=DEV).manual_seed(6), device=DEV).to(torch.bfloat16)
    y = api.gemv_w4(W, d, x)
    q = torch.from_numpy(oracle.int4_unpack(synth.host_u8(W))).double()
    assert torch.equal(y.cpu().double(), q @ x.double().cpu())


@pytest.mark.parametrize("R,K,k", [(151936, 4096, 8), (5003, 1024, 16), (64, 64, 1)])
def test_gemv_w4_topk(cuda_lib, R, K, k):
    W, d, x = _w4(R, K, 7 + k)
    # equal logits: row 11 copies row 40000 (or row 2); a NaN row is never chosen
    src = 40000 if R > 40000 else 2
    W[11] = W[src]
    d[11] = d[src]
    d[5] = float("nan")
    y, ids, vals = api.gemv_w4_topk(W, d, x, k)
    torch.cuda.synchronize()
    yh = y.cpu().numpy().astype(np.float64)
    ref = oracle.gemv_w4(synth.host_u8(W), synth.bits_u16(d), oracle.bf16_to_f64(synth.bits_u16(x)))
    ok = ~np.isnan(ref)
    assert np.isnan(yh[5]) and rel_max_abs(yh[ok], ref[ok]) < GEMV_TOL
    want_ids, want_vals = oracle.topk_first(yh, k)     # the selection rule on the GPU's own logits
    assert list(ids.cpu().numpy()) == list(want_ids)
    np.testing.assert_array_equal(vals.cpu().numpy(), want_vals.astype(np.float32))
    oid, _ = oracle.topk_first(ref, k)
    assert oid[0] == want_ids[0] or abs(ref[oid[0]] - ref[want_ids[0]]) < 1e-4 * np.max(np.abs(ref[ok]))


def test_w4_model_teacher_forced(cuda_lib, parity_log):
    mt = synth.make_model(synth.SMALL_W4, "int4", 51, DEV, ctx=150, steps=8)
    dec = api.Decoder(mt, max_steps=8, top_k=5)
    assert dec.launches_per_step == 1 + 5 * mt.shape.n_layers + 1
    st = teacher_forced(dec, mt, 8, [("bf16", "w4", None, TOL["bf16"])])
    parity_log["w4_small_model"] = st
    assert st["strict"] >= 7
    lg = dec.logits[0].double().cpu().numpy()
    want, _ = oracle.topk_first(lg, 5)
    assert list(dec.topk_ids.cpu().numpy()) == list(want)


def test_w4_qwen3_8b_layer_and_head(cuda_lib, parity_log):
    s = synth.QWEN3_8B
    mt = synth.make_model(s, "int4", 3, DEV, n_layers=1, ctx=4096, steps=1)
    om = oracle_model(mt)
    ks, vs = oracle_caches(mt, 0, 4097)
    dec = api.Decoder(mt, max_steps=1, top_k=8)
    dec.step()
    torch.cuda.synchronize()
    res = dec.residual()[0].double().cpu().numpy()
    x0 = oracle.bf16_to_f64(synth.bits_u16(mt.embed[int(mt.start_tok[0])]))
    ref = oracle.layer_step(om.dims, om.layers[0], x0, ks[0], vs[0], 4096, mode="bf16", act="w4")
    err = rel_max_abs(res, ref)
    assert err < 1e-2
    rows = np.arange(0, s.vocab, 97)
    lg = dec.logits[0].double().cpu().numpy()
    assert rel_max_abs(lg[rows], oracle.lm_head_rows(om, res, rows, act="w4")) < 1e-4
    want, _ = oracle.topk_first(lg, 8)
    assert list(dec.topk_ids.cpu().numpy()) == list(want) and int(dec.tok[0]) == want[0]
    parity_log["w4_qwen3_8b_layer"] = err
    assert api.check_device_error() == 0
