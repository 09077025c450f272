"""Parity of the whole decode step (qd_decode_step / the captured graph) with the
CPU oracle.

Protocol for greedy tokens (teacher-forced): the oracle follows the GPU's own
token stream. At every step the GPU logits must match the oracle's within the
relative max-abs tolerance (2e-2 for the BF16 path, 5e-3 for the f32-activation
Q8_0 lane, 2e-2 for the dp4a lane), the GPU token must be the argmax of the GPU
logits, and it must equal the oracle's argmax unless the oracle's top-1/top-2
gap is below 4x the step's max-abs logit error (a near tie, logged).
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL, oracle_caches, oracle_model, per_layer_resync, rel_max_abs, teacher_forced
from transformer_decode_step_weight_gb300 import api, synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_tiny_bf16_model_teacher_forced(cuda_lib):
    mt = synth.make_model(synth.TINY, "bf16", 1, DEV, ctx=20, steps=12)
    dec = api.Decoder(mt, max_steps=12)
    st = teacher_forced(dec, mt, 12, [("bf16", "bf16", None, TOL["bf16"])])
    assert st["strict"] >= 11
    assert int(dec.pos[0]) == 32 and int(dec.step_ctr[0]) == 12


@pytest.mark.parametrize("act,lane,lm_act,lm_lane", [("f32", api.QD_ACT_F32, None, None),
                                                     ("i8", api.QD_ACT_I8, None, None),
                                                     ("i8", api.QD_ACT_I8, "f32", api.QD_ACT_F32)])
def test_tiny_q8_model_teacher_forced(cuda_lib, act, lane, lm_act, lm_lane):
    # deq = 2 (f32 activations everywhere), 0 (dp4a everywhere) and 1 (dp4a in the
    # layers, the LM head on f32 activations)
    mt = synth.make_model(synth.TINY, "q8_0", 2, DEV, ctx=40, steps=8)
    dec = api.Decoder(mt, max_steps=8, act=lane, lm_act=lm_lane)
    st = teacher_forced(dec, mt, 8, [("f32", act, lm_act, TOL[act])])
    assert st["strict"] >= 7


def test_small_bf16_batch_paged_teacher_forced(cuda_lib):
    # batch 3, 16-token pages through a random page table; every sequence checked
    mt = synth.make_model(synth.SMALL, "bf16", 3, DEV, batch=3, ctx=[70, 129, 300], steps=6, paged=True)
    om = oracle_model(mt)
    caches = [oracle_caches(mt, b, int(mt.seq_lens[b]) + 6) for b in range(3)]
    dec = api.Decoder(mt, max_steps=6)
    toks = [int(t) for t in mt.start_tok]
    for t in range(6):
        dec.step()
        torch.cuda.synchronize()
        for b in range(3):
            g = dec.logits[b].double().cpu().numpy()
            ref = oracle.decode_token(om, toks[b], int(mt.seq_lens[b]) + t, caches[b][0], caches[b][1], mode="bf16",
                                      act="bf16")
            assert rel_max_abs(g, ref) < TOL["bf16"]
            toks[b] = int(dec.tok[b])
            assert toks[b] == oracle.argmax_first(g)
    assert api.check_device_error() == 0


@pytest.mark.parametrize("batch", [3, 8, 12, 64])
def test_batched_tensor_core_step_teacher_forced(cuda_lib, monkeypatch, batch):
    # 3..64 sequences (dims multiples of 64): projections on tcgen05 (below 9 only with
    # QD_SMALLB_IMPL=tc), paged KV through a random page table
    monkeypatch.setenv("QD_SMALLB_IMPL", "tc")
    mt = synth.make_model(synth.SMALL64, "bf16", 7, DEV, batch=batch, ctx=None, steps=3, paged=True)
    om = oracle_model(mt)
    check = sorted({0, batch // 3, batch - 1})
    caches = {b: oracle_caches(mt, b, int(mt.seq_lens[b]) + 3) for b in check}
    dec = api.Decoder(mt, max_steps=3)
    assert dec.launches_per_step == 1 + 8 * 2 + 3
    toks = {b: int(mt.start_tok[b]) for b in check}
    for t in range(3):
        dec.step()
        torch.cuda.synchronize()
        for b in check:
            g = dec.logits[b].double().cpu().numpy()
            ref = oracle.decode_token(om, toks[b], int(mt.seq_lens[b]) + t, caches[b][0], caches[b][1],
                                      mode="bf16", act="bf16")
            assert rel_max_abs(g, ref) < TOL["bf16"], (t, b)
            toks[b] = int(dec.tok[b])
            assert toks[b] == oracle.argmax_first(g)
    assert api.check_device_error() == 0


@pytest.mark.parametrize("shape,batch,norm_rows", [("SMALL64", 2, 1), ("SMALL", 5, 1), ("SMALL64", 8, 1),
                                                    ("TINY", 7, 1), ("SMALL64", 3, 0), ("SMALL", 8, 0)])
def test_small_batch_mma_step_teacher_forced(cuda_lib, monkeypatch, shape, batch, norm_rows):
    # 2..8 sequences: every projection on the mma.sync GEMV (SwiGLU epilogue), the
    # RMSNorms as row kernels (seven launches per layer) or, with QD_MMA_NORM_ROWS=0, in
    # the GEMV prologues (five); paged KV through a random page table
    monkeypatch.setenv("QD_MMA_NORM_ROWS", str(norm_rows))
    mt = synth.make_model(getattr(synth, shape), "bf16", 17 + batch, DEV, batch=batch, ctx=None, steps=3,
                          paged=True)
    om = oracle_model(mt)
    check = sorted({0, batch // 2, batch - 1})
    caches = {b: oracle_caches(mt, b, int(mt.seq_lens[b]) + 3) for b in check}
    dec = api.Decoder(mt, max_steps=3)
    L = mt.shape.n_layers
    assert dec.launches_per_step == (1 + 7 * L + 3 if norm_rows else 1 + 5 * L + 2)
    toks = {b: int(mt.start_tok[b]) for b in check}
    for t in range(3):
        dec.step()
        torch.cuda.synchronize()
        for b in check:
            g = dec.logits[b].double().cpu().numpy()
            ref = oracle.decode_token(om, toks[b], int(mt.seq_lens[b]) + t, caches[b][0], caches[b][1],
                                      mode="bf16", act="bf16")
            assert rel_max_abs(g, ref) < TOL["bf16"], (t, b)
            toks[b] = int(dec.tok[b])
            assert toks[b] == oracle.argmax_first(g)
    assert api.check_device_error() == 0


@pytest.mark.parametrize("batch", [3, 16])
def test_batched_q8_step_teacher_forced(cuda_lib, batch, parity_log):
    # Q8_0 weights (LM head too) at batch > 1: every projection a tcgen05 GEMM with the
    # weights widened to bf16 on chip; paged KV through a random page table. Held to
    # the pages' Q8_0 definition (w = f32(d) q, act "f32" on the bf16 activations) and,
    # as a diagnostic, to the lane that widens each weight to bf16 as the kernel does.
    mt = synth.make_model(synth.SMALL256, "q8_0", 8, DEV, batch=batch, ctx=None, steps=3, paged=True)
    om = oracle_model(mt)
    check = sorted({0, batch // 2, batch - 1})
    lanes = ("f32", "w_bf16")
    caches = {(b, a): oracle_caches(mt, b, int(mt.seq_lens[b]) + 3) for b in check for a in lanes}
    dec = api.Decoder(mt, max_steps=3)
    assert dec.launches_per_step == 1 + 8 * 2 + 3
    toks = {b: int(mt.start_tok[b]) for b in check}
    worst = {a: 0.0 for a in lanes}
    for t in range(3):
        dec.step()
        torch.cuda.synchronize()
        for b in check:
            g = dec.logits[b].double().cpu().numpy()
            for a in lanes:
                kc, vc = caches[(b, a)]
                ref = oracle.decode_token(om, toks[b], int(mt.seq_lens[b]) + t, kc, vc, mode="bf16", act=a)
                err = rel_max_abs(g, ref)
                worst[a] = max(worst[a], err)
                assert err < TOL["w_bf16"], (t, b, a, err)
            toks[b] = int(dec.tok[b])
            assert toks[b] == oracle.argmax_first(g)
    parity_log[f"batched_q8_step_b{batch}"] = {"vs_q8_0_definition": worst["f32"], "vs_widened_lane": worst["w_bf16"]}
    assert api.check_device_error() == 0


@pytest.mark.parametrize("wtype,acts,batch", [("bf16", ("bf16",), 64), ("bf16", ("bf16",), 8),
                                              ("q8_0", ("f32", "w_bf16"), 64)])
def test_qwen3_8b_batched_paged_layer(cuda_lib, wtype, acts, batch, parity_log):
    """The batched workload's shapes: 64 sequences (and 8, on the mma.sync GEMV), Qwen3-8B
    layer, 16-token pages through a random page table, context uniform in [128, 4096];
    sampled sequences checked whole. Q8_0: held to the pages' Q8_0 definition ("f32", on
    the bf16 activations) and to the widened-weight lane."""
    s = synth.QWEN3_8B
    mt = synth.make_model(s, wtype, 9, DEV, n_layers=1, batch=batch, ctx=None, steps=1, paged=True)
    om = oracle_model(mt)
    dec = api.Decoder(mt, max_steps=1)
    check = sorted({0, batch // 2 - 1, batch - 1})
    dec.step()
    torch.cuda.synchronize()
    res = dec.residual()
    worst = {}
    for act in acts:
        caches = {b: oracle_caches(mt, b, int(mt.seq_lens[b]) + 1) for b in check}
        for b in check:
            x0 = oracle.bf16_to_f64(synth.bits_u16(mt.embed[int(mt.start_tok[b])]))
            ref = oracle.layer_step(om.dims, om.layers[0], x0, caches[b][0][0], caches[b][1][0],
                                    int(mt.seq_lens[b]), mode="bf16", act=act)
            err = rel_max_abs(res[b].double().cpu().numpy(), ref)
            worst[f"layer/{act}"] = max(worst.get(f"layer/{act}", 0.0), err)
            assert err < TOL[act if act != "f32" else "w_bf16"], (b, act, err)
        rows = np.arange(0, s.vocab, 211)
        for b in check:
            lg = dec.logits[b].double().cpu().numpy()
            ref = oracle.lm_head_rows(om, res[b].double().cpu().numpy(), rows, act=act)
            err = rel_max_abs(lg[rows], ref)
            worst[f"lm_head/{act}"] = max(worst.get(f"lm_head/{act}", 0.0), err)
            assert err < TOL[act if act != "f32" else "w_bf16"], (b, act, err)
            assert int(dec.tok[b]) == oracle.argmax_first(lg)
    parity_log[f"qwen3_8b_batched_paged_layer/{wtype}/b{batch}"] = worst
    assert api.check_device_error() == 0


def test_graph_replay_is_bit_identical_to_eager(cuda_lib):
    runs = []
    for use_graph in (False, True):
        mt = synth.make_model(synth.SMALL, "bf16", 4, DEV, ctx=100, steps=8)
        dec = api.Decoder(mt, max_steps=8)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            if use_graph:
                dec.capture(4)
                addr = (dec.tok.data_ptr(), dec.pos.data_ptr(), dec.logits.data_ptr())
                dec.replay()
                dec.replay()
                assert addr == (dec.tok.data_ptr(), dec.pos.data_ptr(), dec.logits.data_ptr())
            else:
                for _ in range(8):
                    dec.step()
        s.synchronize()
        runs.append((dec.out_tokens.clone(), dec.logits.clone(), mt.k_cache[0].clone(), dec.pos.clone()))
        dec.close()
    for a, b in zip(runs[0], runs[1]):
        assert torch.equal(a, b)
    assert int(runs[1][3][0]) == 108


def test_qwen3_06b_layer_workload(cuda_lib):
    """One Qwen3-0.6B-shaped layer at position 128 over a 128-token cache; input hidden ~ N(0, 1)."""
    s = synth.QWEN3_06B
    mt = synth.make_model(s, "bf16", 0, DEV, n_layers=1, ctx=128, steps=1)
    hid = synth.make_hidden(0, s.hidden, DEV)
    tok = int(mt.start_tok[0])
    mt.embed[tok] = hid[0].to(torch.bfloat16)    # the layer input is this hidden state (bf16 storage)
    om = oracle_model(mt)
    ks, vs = oracle_caches(mt, 0, 129)
    dec = api.Decoder(mt, max_steps=1)
    dec.step()
    torch.cuda.synchronize()
    res = dec.residual()[0].double().cpu().numpy()
    x0 = oracle.bf16_to_f64(synth.bits_u16(mt.embed[tok]))
    ref = oracle.layer_step(om.dims, om.layers[0], x0, ks[0], vs[0], 128, mode="bf16", act="bf16")
    assert rel_max_abs(res, ref) < 2e-3
    # the K/V rows written at slot 128 (bf16) against the oracle's
    k_gpu = oracle.bf16_to_f64(synth.bits_u16(mt.k_cache[0][0, :, 128, :]))
    v_gpu = oracle.bf16_to_f64(synth.bits_u16(mt.v_cache[0][0, :, 128, :]))
    assert rel_max_abs(k_gpu, ks[0][:, 128]) < 1e-2
    assert rel_max_abs(v_gpu, vs[0][:, 128]) < 1e-2
    # LM head on the GPU's own final residual: sampled rows + the argmax
    rows = np.arange(0, s.vocab, 37)
    lg = dec.logits[0].double().cpu().numpy()
    assert rel_max_abs(lg[rows], oracle.lm_head_rows(om, res, rows)) < 1e-3


@pytest.mark.parametrize("wtype,act", [("bf16", "bf16"), ("q8_0", "f32"), ("q8_0", "i8")])
def test_qwen3_8b_full_size_layer_and_head(cuda_lib, wtype, act):
    """Full Qwen3-8B shapes in the launch configuration the bench uses: one layer at
    context 4096 (2048 for Q8_0) checked whole, the 151936-row LM head sampled."""
    s = synth.QWEN3_8B
    ctx = 4096 if wtype == "bf16" else 2048
    mt = synth.make_model(s, wtype, 3, DEV, n_layers=1, ctx=ctx, steps=1)
    om = oracle_model(mt)
    ks, vs = oracle_caches(mt, 0, ctx + 1)
    lane = api.QD_ACT_I8 if act == "i8" else api.QD_ACT_F32
    dec = api.Decoder(mt, max_steps=1, act=lane)
    dec.step()
    torch.cuda.synchronize()
    res = dec.residual()[0].double().cpu().numpy()
    mode = "bf16" if wtype == "bf16" else "f32"
    x0 = oracle.bf16_to_f64(synth.bits_u16(mt.embed[int(mt.start_tok[0])]))
    ref = oracle.layer_step(om.dims, om.layers[0], x0, ks[0], vs[0], ctx, mode=mode, act=act)
    assert rel_max_abs(res, ref) < TOL[act]
    rows = np.arange(0, s.vocab, 101)
    lg = dec.logits[0].double().cpu().numpy()
    assert rel_max_abs(lg[rows], oracle.lm_head_rows(om, res, rows, mode=mode, act=act)) < TOL[act]
    assert int(dec.tok[0]) == oracle.argmax_first(lg)
    assert api.check_device_error() == 0


def test_qwen3_06b_model_teacher_forced(cuda_lib, parity_log):
    """Qwen3-0.6B-shaped model (28 layers, tied head) at context 2048: every layer on the
    GPU's own input, then 16 greedy steps teacher-forced (end-to-end limit from the
    oracle's own accumulation drift, as in test_gpu_model)."""
    mt = synth.make_model(synth.QWEN3_06B, "bf16", 5, DEV, ctx=2048, steps=16)
    layers = per_layer_resync(mt, api.QD_ACT_F32, "bf16", "bf16", tol=1e-2)
    dec = api.Decoder(mt, max_steps=16)
    st = teacher_forced(dec, mt, 16, [("bf16", "bf16", None, TOL["bf16"])], floor_factor=3.0, lm_resync=True)
    st["per_layer_worst"] = layers
    parity_log["qwen3_06b_model"] = st
    assert st["strict"] >= 12


# ---------------------------------------------------------------- the persistent step kernel
# QD_STEP_PATH=persistent runs a batch-1 BF16 step as one persistent kernel (the whole
# step's weight stream through one ring per SM, phases joined by counters in global
# memory). The library reads the variable on every call.


@pytest.fixture
def persistent(monkeypatch):
    monkeypatch.setenv("QD_STEP_PATH", "persistent")


def test_persistent_step_tiny_and_small_teacher_forced(cuda_lib, persistent):
    for shape, ctx, steps in ((synth.TINY, 20, 12), (synth.SMALL, 300, 6), (synth.SMALL64, 77, 5)):
        mt = synth.make_model(shape, "bf16", 11, DEV, ctx=ctx, steps=steps)
        dec = api.Decoder(mt, max_steps=steps)
        assert dec.launches_per_step == 1
        st = teacher_forced(dec, mt, steps, [("bf16", "bf16", None, TOL["bf16"])])
        assert st["strict"] >= steps - 1, shape.name
        dec.close()


def test_persistent_step_matches_kernel_path(cuda_lib, monkeypatch):
    # the same model and start state through both paths: logits within the parity
    # tolerance of each other, and the persistent path is deterministic
    outs = {}
    for path in ("kernels", "persistent", "persistent"):
        monkeypatch.setenv("QD_STEP_PATH", path)
        mt = synth.make_model(synth.SMALL, "bf16", 12, DEV, ctx=500, steps=4)
        dec = api.Decoder(mt, max_steps=4)
        for _ in range(4):
            dec.step()
        torch.cuda.synchronize()
        outs.setdefault(path, []).append((dec.logits.clone(), dec.out_tokens.clone(), mt.k_cache[1].clone()))
        dec.close()
    a, b = outs["kernels"][0], outs["persistent"][0]
    assert rel_max_abs(b[0].double().cpu().numpy(), a[0].double().cpu().numpy()) < 2e-2
    for x, y in zip(outs["persistent"][0], outs["persistent"][1]):
        assert torch.equal(x, y)
    assert api.check_device_error() == 0


def test_persistent_graph_replay_is_bit_identical_to_eager(cuda_lib, persistent):
    runs = []
    for use_graph in (False, True):
        mt = synth.make_model(synth.SMALL, "bf16", 4, DEV, ctx=100, steps=8)
        dec = api.Decoder(mt, max_steps=8)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            if use_graph:
                dec.capture(4)
                dec.replay()
                dec.replay()
            else:
                for _ in range(8):
                    dec.step()
        s.synchronize()
        runs.append((dec.out_tokens.clone(), dec.logits.clone(), mt.k_cache[0].clone(), dec.pos.clone()))
        dec.close()
    for a, b in zip(runs[0], runs[1]):
        assert torch.equal(a, b)
    assert api.check_device_error() == 0


def test_persistent_step_qwen3_8b_full_size_layer_and_head(cuda_lib, persistent):
    s = synth.QWEN3_8B
    mt = synth.make_model(s, "bf16", 3, DEV, n_layers=1, ctx=4096, steps=1)
    om = oracle_model(mt)
    ks, vs = oracle_caches(mt, 0, 4097)
    dec = api.Decoder(mt, max_steps=1)
    assert dec.launches_per_step == 1
    dec.step()
    torch.cuda.synchronize()
    res = dec.residual()[0].double().cpu().numpy()
    x0 = oracle.bf16_to_f64(synth.bits_u16(mt.embed[int(mt.start_tok[0])]))
    ref = oracle.layer_step(om.dims, om.layers[0], x0, ks[0], vs[0], 4096, mode="bf16", act="bf16")
    assert rel_max_abs(res, ref) < 1e-2
    rows = np.arange(0, s.vocab, 101)
    lg = dec.logits[0].double().cpu().numpy()
    assert rel_max_abs(lg[rows], oracle.lm_head_rows(om, res, rows)) < 1e-3
    assert int(dec.tok[0]) == oracle.argmax_first(lg)
    assert api.check_device_error() == 0
