"""Prefill (qd_prefill) against the oracle run one token at a time.

"qwen3-8b-rtx4080-cutedsl" README, "Flash Attention 2" / "Baseline tiled GEMM": the
prompt's n tokens pass through each layer as one batch of rows, with causal
attention among them. Row i must give exactly what a plain decode step gives for
token i after tokens 0 .. i - 1, so the oracle decodes the prompt token by token
(decode_token writes each K/V row before the next token reads it); the last row's
logits, every K/V row written to the cache, the argmax and the state advance are
checked, and decoding continues from the prefilled cache.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL, oracle_caches, oracle_model, rel_max_abs
from transformer_decode_step_weight_gb300 import api, synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _prompt(mt, n, seed):
    return [int(t) for t in np.random.default_rng(seed).integers(0, mt.shape.vocab, n)]


def _oracle_prefill(om, mt, tokens, pos0, act="bf16", mode="bf16", extra=0, trace=None):
    ks, vs = oracle_caches(mt, 0, pos0 + len(tokens) + extra)
    last = None
    for i, t in enumerate(tokens):
        tr = [] if trace is not None else None
        last = oracle.decode_token(om, t, pos0 + i, ks, vs, mode=mode, act=act, residual_trace=tr)
        if trace is not None:
            trace.append(tr)
    return last, ks, vs


def _check_kv(mt, ks, vs, p, n, tol=2e-2):
    for li in range(len(mt.layers)):
        for cache, ref in ((mt.k_cache[li], ks[li]), (mt.v_cache[li], vs[li])):
            got = oracle.bf16_to_f64(oracle.gather_paged(synth.bits_u16(cache), mt.page_table[0].cpu().numpy(),
                                                         p + n))
            assert rel_max_abs(got[:, p:p + n], ref[:, p:p + n]) < tol, li


# QD_PREFILL_P_HILO: the mma.sync attention's P as bf16 hi + lo (1) or its bf16 value
# alone (0); QD_PREFILL_ATTN=tc: the tcgen05 attention (128-row query tiles: ragged
# tiles at 1, 63, 130 and 1030 rows)
@pytest.mark.parametrize("n,hilo,attn", [(1, 1, "mma"), (63, 1, "mma"), (130, 1, "mma"), (1030, 1, "mma"),
                                         (130, 0, "mma"), (1030, 0, "mma"), (1, 1, "tc"), (63, 1, "tc"),
                                         (130, 1, "tc"), (1030, 1, "tc")])
def test_prefill_bf16(cuda_lib, parity_log, monkeypatch, n, hilo, attn):
    monkeypatch.setenv("QD_PREFILL_P_HILO", str(hilo))
    monkeypatch.setenv("QD_PREFILL_ATTN", attn)
    _prefill_case(parity_log, n, f"prefill_bf16_n{n}_hilo{hilo}_{attn}")


# The prefill GEMMs above 128 rows: the persistent kernels (default) and one CTA per
# tile (QD_GEMM_WIDE=tiles). 2100 rows = 9 token tiles (the last ragged); the gate+up
# projection (F = 1408: 22 tiles of 64 gate over 64 up rows) gives 198 items, so CTAs
# take a second item and reuse both accumulators and exchange buffers.
@pytest.mark.parametrize("form", ["persistent", "tiles"])
def test_prefill_bf16_gemm_forms(cuda_lib, parity_log, monkeypatch, form):
    monkeypatch.setenv("QD_GEMM_WIDE", form)
    _prefill_case(parity_log, 2100, f"prefill_bf16_n2100_{form}")


def _prefill_case(parity_log, n, key):
    mt = synth.make_model(synth.SMALL64, "bf16", 60 + n, DEV, ctx=37, steps=n + 4)
    om = oracle_model(mt)
    dec = api.Decoder(mt, max_steps=n + 4, prefill_max=n)
    pos0, step0 = int(mt.seq_lens[0]), int(dec.step_ctr[0])
    toks = _prompt(mt, n, n)
    dec.prefill(torch.tensor(toks, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    ref, ks, vs = _oracle_prefill(om, mt, toks, pos0)
    got = dec.prefill_logits.double().cpu().numpy()
    err = rel_max_abs(got, ref)
    assert err < TOL["bf16"], err
    _check_kv(mt, ks, vs, pos0, n)
    tk = oracle.argmax_first(got)
    assert int(dec.tok[0]) == tk and int(dec.pos[0]) == pos0 + n and int(dec.step_ctr[0]) == step0 + 1
    assert int(dec.out_tokens[0, step0]) == tk
    if oracle.argmax_first(ref) != tk:   # only at a near tie
        top = np.sort(ref)[-2:]
        assert top[1] - top[0] < 4 * np.max(np.abs(got - ref))
    parity_log[key] = err
    assert api.check_device_error() == 0


def test_prefill_then_decode(cuda_lib, parity_log):
    # decoding continues from the prefilled cache: three greedy steps held to the oracle
    n = 90
    mt = synth.make_model(synth.SMALL64, "bf16", 77, DEV, ctx=20, steps=n + 4)
    om = oracle_model(mt)
    dec = api.Decoder(mt, max_steps=n + 4, prefill_max=n)
    pos0 = int(mt.seq_lens[0])
    toks = _prompt(mt, n, 5)
    dec.prefill(torch.tensor(toks, dtype=torch.int32, device=DEV))
    _, ks, vs = _oracle_prefill(om, mt, toks, pos0, extra=3)
    worst = 0.0
    for i in range(3):
        t = int(dec.tok[0])
        dec.step()
        torch.cuda.synchronize()
        ref = oracle.decode_token(om, t, pos0 + n + i, ks, vs)
        err = rel_max_abs(dec.logits[0].double().cpu().numpy(), ref)
        worst = max(worst, err)
        assert err < TOL["bf16"], (i, err)
    parity_log["prefill_then_decode"] = worst
    assert api.check_device_error() == 0


@pytest.mark.parametrize("attn", ["mma", "tc"])
def test_prefill_paged_cache(cuda_lib, monkeypatch, attn):
    # a paged cache (16-token pages through a permuted page table): same logits and
    # K/V as the oracle on the logical sequence
    monkeypatch.setenv("QD_PREFILL_ATTN", attn)
    n = 75
    mt = synth.make_model(synth.SMALL64, "bf16", 88, DEV, batch=1, ctx=None, steps=n + 2, paged=True)
    om = oracle_model(mt)
    dec = api.Decoder(mt, max_steps=n + 2, prefill_max=n)
    pos0 = int(mt.seq_lens[0])
    toks = _prompt(mt, n, 9)
    dec.prefill(torch.tensor(toks, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    ref, ks, vs = _oracle_prefill(om, mt, toks, pos0)
    assert rel_max_abs(dec.prefill_logits.double().cpu().numpy(), ref) < TOL["bf16"]
    _check_kv(mt, ks, vs, pos0, n)
    assert api.check_device_error() == 0


# Q8_0 weights: the rows run on the tensor cores with each weight widened to bf16, in
# the Q8_0 GEMM's converters up to 128 rows and above that by a widening pass ahead of
# the bf16 GEMMs (from 1024 rows the gate+up one with the SwiGLU epilogue); held to the
# pages' Q8_0 definition and to the widened-weight lane
@pytest.mark.parametrize("n", [70, 300, 1030])
def test_prefill_q8_0(cuda_lib, parity_log, n):
    mt = synth.make_model(synth.SMALL256, "q8_0", 45, DEV, ctx=30, steps=n + 2)
    om = oracle_model(mt)
    dec = api.Decoder(mt, max_steps=n + 2, prefill_max=n)
    pos0 = int(mt.seq_lens[0])
    toks = _prompt(mt, n, 3)
    dec.prefill(torch.tensor(toks, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    got = dec.prefill_logits.double().cpu().numpy()
    worst = {}
    for act in ("f32", "w_bf16"):
        ref, _, _ = _oracle_prefill(om, mt, toks, pos0, act=act)
        worst[act] = rel_max_abs(got, ref)
        assert worst[act] < TOL["w_bf16"], (act, worst[act])
    parity_log[f"prefill_q8_0_n{n}"] = worst
    assert api.check_device_error() == 0


@pytest.mark.parametrize("hilo,attn", [(1, "mma"), (0, "mma"), (1, "tc")])
def test_prefill_qwen3_8b_layer(cuda_lib, parity_log, monkeypatch, hilo, attn):
    """Full Qwen3-8B shapes: one layer after a 4096-token cache, a 70-token prompt;
    sampled rows' residuals whole, every K/V row, and sampled LM-head rows."""
    monkeypatch.setenv("QD_PREFILL_P_HILO", str(hilo))
    monkeypatch.setenv("QD_PREFILL_ATTN", attn)
    s = synth.QWEN3_8B
    n = 70
    mt = synth.make_model(s, "bf16", 5, DEV, n_layers=1, ctx=4096, steps=n)
    om = oracle_model(mt)
    dec = api.Decoder(mt, max_steps=n, prefill_max=n)
    toks = _prompt(mt, n, 1)
    dec.prefill(torch.tensor(toks, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    res = dec.rows_residual(n).double().cpu().numpy()
    ks, vs = oracle_caches(mt, 0, 4096 + n)
    worst = 0.0
    for i, t in enumerate(toks):
        x0 = oracle.bf16_to_f64(synth.bits_u16(mt.embed[t]))
        ref = oracle.layer_step(om.dims, om.layers[0], x0, ks[0], vs[0], 4096 + i, mode="bf16", act="bf16")
        if i in (0, 31, 63, 64, n - 1):
            err = rel_max_abs(res[i], ref)
            worst = max(worst, err)
            assert err < 1e-2, (i, err)
    _check_kv(mt, ks, vs, 4096, n)
    rows = np.arange(0, s.vocab, 211)
    lg = dec.prefill_logits.double().cpu().numpy()
    assert rel_max_abs(lg[rows], oracle.lm_head_rows(om, res[n - 1], rows)) < 1e-3
    assert int(dec.tok[0]) == oracle.argmax_first(lg)
    parity_log[f"prefill_qwen3_8b_layer_hilo{hilo}_{attn}"] = worst
    assert api.check_device_error() == 0


def test_prefill_rejects_bad_arguments(cuda_lib):
    mt = synth.make_model(synth.SMALL64, "bf16", 2, DEV, ctx=10, steps=8)
    dec = api.Decoder(mt, max_steps=8, prefill_max=8)
    with pytest.raises(api.QDError):
        dec.prefill(torch.zeros(0, dtype=torch.int32, device=DEV))
    with pytest.raises(api.QDError):        # more rows than the workspace was sized for
        dec.prefill(torch.zeros(4000, dtype=torch.int32, device=DEV))
    w4 = synth.make_model(synth.SMALL_W4, "int4", 2, DEV, ctx=10, steps=8)
    d4 = api.Decoder(w4, max_steps=8, prefill_max=8)
    with pytest.raises(api.QDError):
        d4.prefill(torch.zeros(4, dtype=torch.int32, device=DEV))
    # a prompt that runs past the cache: the position error bit, nothing written out of range
    dec2 = api.Decoder(mt, max_steps=8, prefill_max=64)
    dec2.prefill(torch.zeros(64, dtype=torch.int32, device=DEV))
    assert api.check_device_error() & 2   # QD_DEVERR_POS
