"""Speculative verify (qd_verify_step) against the oracle.

"qwen3-8b-rtx4080-cutedsl" README, "Speculative decoding": the target model checks
k drafted tokens in one forward pass. The pass is k rows of one sequence at
positions pos .. pos + k - 1 with causal attention among them, so row i must give
exactly what a plain decode step gives for input i after inputs 0 .. i - 1: the
oracle runs the inputs one token at a time (decode_token writes each K/V row before
the next token reads it), and every row's logits, the K/V rows written to the
cache, the per-row argmax, the accepted prefix and the state advance are checked.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL, oracle_caches, oracle_model, rel_max_abs
from transformer_decode_step_weight_gb300 import api, synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _oracle_run(om, mt, history, inputs, pos0, act="bf16", mode="bf16"):
    """The oracle over `history` (tokens already at positions pos0 ..) then `inputs`:
    the logits of each input, and the caches afterwards."""
    n = len(history) + len(inputs)
    ks, vs = oracle_caches(mt, 0, pos0 + n)
    for i, t in enumerate(history):
        oracle.decode_token(om, t, pos0 + i, ks, vs, mode=mode, act=act)
    p = pos0 + len(history)
    rows = [oracle.decode_token(om, t, p + i, ks, vs, mode=mode, act=act) for i, t in enumerate(inputs)]
    return rows, ks, vs


def _check_pass(dec, mt, om, history, draft, pos0, step0, acts, tol, mode="bf16"):
    """Check the pass just run: inputs tok, draft at position pos0 + len(history)."""
    k = len(draft) + 1
    p = pos0 + len(history)
    inputs = [int(dec.out_tokens[0, step0 - 1]) if step0 else int(mt.start_tok[0])] + list(draft)
    g = dec.verify_logits[:k].double().cpu().numpy()
    tgt = [int(t) for t in dec.verify_target[:k].cpu()]
    for i in range(k):
        assert tgt[i] == oracle.argmax_first(g[i]), i
    worst = {}
    for act in acts:
        refs, ks, vs = _oracle_run(om, mt, history, inputs, pos0, act=act, mode=mode)
        for i in range(k):
            err = rel_max_abs(g[i], refs[i])
            worst[act] = max(worst.get(act, 0.0), err)
            assert err < tol, (act, i, err)
            otok = oracle.argmax_first(refs[i])
            if otok != tgt[i]:   # only at a near tie
                top = np.sort(refs[i])[-2:]
                assert top[1] - top[0] < 4 * np.max(np.abs(g[i] - refs[i])), (i, tgt[i], otok)
    # the K/V rows of the k inputs in the cache (contiguous cache: page 0, slots p ..)
    for li in range(len(mt.layers)):
        for cache, ref in ((mt.k_cache[li], ks[li]), (mt.v_cache[li], vs[li])):
            got = oracle.bf16_to_f64(synth.bits_u16(cache[0, :, p:p + k, :]))
            assert rel_max_abs(got, ref[:, p:p + k]) < 2e-2, li
    m = 0
    while m < k - 1 and draft[m] == tgt[m]:
        m += 1
    assert int(dec.n_accept[0]) == m
    assert int(dec.tok[0]) == tgt[m] and int(dec.pos[0]) == p + m + 1 and int(dec.step_ctr[0]) == step0 + m + 1
    emitted = [int(t) for t in dec.out_tokens[0, step0:step0 + m + 1].cpu()]
    assert emitted == list(draft[:m]) + [tgt[m]]
    return inputs[:m + 1], m, worst


def _greedy(om, mt, history, tok, pos0, n, act="bf16", mode="bf16"):
    """The oracle's own greedy continuation of `tok` after `history` (n tokens)."""
    ks, vs = oracle_caches(mt, 0, pos0 + len(history) + n)
    for i, t in enumerate(history):
        oracle.decode_token(om, t, pos0 + i, ks, vs, mode=mode, act=act)
    out, cur = [], tok
    for i in range(n):
        cur = oracle.argmax_first(oracle.decode_token(om, cur, pos0 + len(history) + i, ks, vs, mode=mode, act=act))
        out.append(cur)
    return out


# QD_SMALLB_IMPL: "mma" (default) runs the pass's projections on the mma.sync GEMV,
# "tc" on the tcgen05 GEMMs
@pytest.mark.parametrize("k,impl", [(2, "mma"), (4, "mma"), (8, "mma"), (4, "tc"), (8, "tc")])
def test_verify_teacher_forced_bf16(cuda_lib, parity_log, monkeypatch, k, impl):
    monkeypatch.setenv("QD_SMALLB_IMPL", impl)
    mt = synth.make_model(synth.SMALL64, "bf16", 21 + k, DEV, ctx=100, steps=2 * k + 2)
    om = oracle_model(mt)
    dec = api.Decoder(mt, max_steps=2 * k + 2, verify_k=k)
    pos0 = int(mt.seq_lens[0])
    # pass 1: random drafts (almost surely rejected at once)
    draft = [int(t) for t in np.random.default_rng(k).integers(0, mt.shape.vocab, k - 1)]
    dec.verify(torch.tensor(draft, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    hist, m1, w1 = _check_pass(dec, mt, om, [], draft, pos0, 0, ["bf16"], TOL["bf16"])
    # pass 2: drafts that follow the oracle's greedy continuation (accepted but at a near tie)
    step1 = int(dec.step_ctr[0])
    draft = _greedy(om, mt, hist, int(dec.tok[0]), pos0, k - 1)
    dec.verify(torch.tensor(draft, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    _, m2, w2 = _check_pass(dec, mt, om, hist, draft, pos0, step1, ["bf16"], TOL["bf16"])
    assert m2 >= k - 2
    parity_log[f"verify_bf16_k{k}_{impl}"] = {"accepted": [m1, m2], "worst_rel_err": max(w1["bf16"], w2["bf16"])}
    assert api.check_device_error() == 0


@pytest.mark.parametrize("k", [3, 8])
def test_verify_paged_cache(cuda_lib, k):
    # 16-token pages through a random page table: the pass's shared-K/V attention
    # follows the sequence's page-table row; every row's logits and argmax against
    # the oracle
    mt = synth.make_model(synth.SMALL64, "bf16", 51 + k, DEV, ctx=[333], steps=k + 1, paged=True)
    om = oracle_model(mt)
    dec = api.Decoder(mt, max_steps=k + 1, verify_k=k)
    draft = [int(t) for t in np.random.default_rng(k).integers(0, mt.shape.vocab, k - 1)]
    dec.verify(torch.tensor(draft, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    inputs = [int(mt.start_tok[0])] + draft
    refs, _, _ = _oracle_run(om, mt, [], inputs, int(mt.seq_lens[0]))
    g = dec.verify_logits[:k].double().cpu().numpy()
    for i in range(k):
        assert rel_max_abs(g[i], refs[i]) < TOL["bf16"], i
        assert int(dec.verify_target[i]) == oracle.argmax_first(g[i])
    assert api.check_device_error() == 0


def test_verify_equals_greedy_steps(cuda_lib):
    # drafts = the GPU's own next greedy tokens: all accepted, and the state and tokens
    # are those of k plain greedy steps
    k = 6
    mt = synth.make_model(synth.SMALL64, "bf16", 31, DEV, ctx=200, steps=k)
    ref = api.Decoder(mt, max_steps=k)
    for _ in range(k):
        ref.step()
    torch.cuda.synchronize()
    toks = [int(t) for t in ref.out_tokens[0].cpu()]
    ref_logits = ref.logits.clone()
    ref.close()
    dec = api.Decoder(mt, max_steps=k, verify_k=k)
    dec.verify(torch.tensor(toks[:k - 1], dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert int(dec.n_accept[0]) == k - 1
    assert [int(t) for t in dec.verify_target.cpu()] == toks
    assert [int(t) for t in dec.out_tokens[0].cpu()] == toks
    assert int(dec.pos[0]) == int(mt.seq_lens[0]) + k and int(dec.tok[0]) == toks[-1]
    assert rel_max_abs(dec.verify_logits[k - 1].double().cpu().numpy(), ref_logits[0].double().cpu().numpy()) < 2e-2
    assert api.check_device_error() == 0


def test_verify_then_decode(cuda_lib):
    # a verify pass leaves the decode step's workspace as it was: greedy steps after it
    # follow the oracle from the cache the pass wrote
    k = 4
    mt = synth.make_model(synth.SMALL64, "bf16", 13, DEV, ctx=50, steps=k + 3)
    om = oracle_model(mt)
    dec = api.Decoder(mt, max_steps=k + 3, verify_k=k)
    pos0 = int(mt.seq_lens[0])
    draft = [int(t) for t in np.random.default_rng(4).integers(0, mt.shape.vocab, k - 1)]
    dec.verify(torch.tensor(draft, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    m = int(dec.n_accept[0])
    hist = ([int(mt.start_tok[0])] + draft)[:m + 1]
    ks, vs = oracle_caches(mt, 0, pos0 + m + 1 + 2)
    for i, t in enumerate(hist):
        oracle.decode_token(om, t, pos0 + i, ks, vs)
    for i in range(2):
        t = int(dec.tok[0])
        dec.step()
        torch.cuda.synchronize()
        ref = oracle.decode_token(om, t, pos0 + m + 1 + i, ks, vs)
        assert rel_max_abs(dec.logits[0].double().cpu().numpy(), ref) < TOL["bf16"], i
    assert api.check_device_error() == 0


@pytest.mark.parametrize("impl", ["mma", "tc"])
def test_verify_qwen3_8b_layer_k8(cuda_lib, parity_log, monkeypatch, impl):
    """Full Qwen3-8B shapes: one layer at context 4096 and the 151936-row LM head, k = 8
    rows, each row's residual checked whole and its LM-head rows sampled."""
    monkeypatch.setenv("QD_SMALLB_IMPL", impl)
    s = synth.QWEN3_8B
    k = 8
    mt = synth.make_model(s, "bf16", 3, DEV, n_layers=1, ctx=4096, steps=k)
    om = oracle_model(mt)
    dec = api.Decoder(mt, max_steps=k, verify_k=k)
    draft = [int(t) for t in np.random.default_rng(8).integers(0, s.vocab, k - 1)]
    dec.verify(torch.tensor(draft, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    inputs = [int(mt.start_tok[0])] + draft
    res = dec.rows_residual(k).double().cpu().numpy()
    ks, vs = oracle_caches(mt, 0, 4096 + k)
    rows = np.arange(0, s.vocab, 211)
    worst = 0.0
    for i, t in enumerate(inputs):
        x0 = oracle.bf16_to_f64(synth.bits_u16(mt.embed[t]))
        ref = oracle.layer_step(om.dims, om.layers[0], x0, ks[0], vs[0], 4096 + i, mode="bf16", act="bf16")
        err = rel_max_abs(res[i], ref)
        worst = max(worst, err)
        assert err < 1e-2, (i, err)
        lg = dec.verify_logits[i].double().cpu().numpy()
        assert rel_max_abs(lg[rows], oracle.lm_head_rows(om, res[i], rows)) < 1e-3
        assert int(dec.verify_target[i]) == oracle.argmax_first(lg)
    parity_log[f"verify_qwen3_8b_layer_k8_{impl}"] = worst
    assert api.check_device_error() == 0


def test_verify_q8_0(cuda_lib, parity_log):
    # Q8_0 weights: the rows run on the tensor cores with each weight widened to bf16;
    # held to the pages' Q8_0 definition and to the widened-weight lane
    k = 4
    mt = synth.make_model(synth.SMALL256, "q8_0", 41, DEV, ctx=90, steps=k + 1)
    om = oracle_model(mt)
    dec = api.Decoder(mt, max_steps=k + 1, verify_k=k)
    draft = [int(t) for t in np.random.default_rng(3).integers(0, mt.shape.vocab, k - 1)]
    dec.verify(torch.tensor(draft, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    _, _, w = _check_pass(dec, mt, om, [], draft, int(mt.seq_lens[0]), 0, ["f32", "w_bf16"], TOL["w_bf16"])
    parity_log["verify_q8_0_k4"] = w
    assert api.check_device_error() == 0


def test_verify_rejects_bad_arguments(cuda_lib, monkeypatch):
    mt = synth.make_model(synth.SMALL64, "bf16", 1, DEV, ctx=10, steps=4)
    dec = api.Decoder(mt, max_steps=4, verify_k=4)
    with pytest.raises(api.QDError):
        dec.verify(torch.zeros(8, dtype=torch.int32, device=DEV))    # k = 9 > 8
    # K = 1376: a multiple of 32 (the mma.sync GEMV takes it), not of 64 (the tcgen05 GEMM)
    monkeypatch.setenv("QD_SMALLB_IMPL", "tc")
    bad = synth.make_model(synth.SMALL, "bf16", 1, DEV, ctx=10, steps=4)
    d2 = api.Decoder(bad, max_steps=4, verify_k=4)
    with pytest.raises(api.QDError):
        d2.verify(torch.zeros(3, dtype=torch.int32, device=DEV))


def test_verify_past_the_cache_flags_the_position(cuda_lib):
    # a pass whose rows run past the cache: K/V write, attention and its merge skip the
    # rows out of range and the position error bit is set (nothing written out of range)
    mt = synth.make_model(synth.SMALL64, "bf16", 7, DEV, ctx=20, steps=4)
    dec = api.Decoder(mt, max_steps=4, verify_k=8)
    before = [c.clone() for c in mt.k_cache]
    dec.verify(torch.zeros(7, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert api.check_device_error() & 2   # QD_DEVERR_POS
    # the cached rows below the pass's first position are untouched
    for b, a in zip(before, mt.k_cache):
        assert torch.equal(b[..., :20, :], a[..., :20, :])


def test_verify_k_not_multiple_of_64_on_mma(cuda_lib):
    # the same K = 1376 model on the mma.sync GEMV: the pass runs and matches the oracle
    k = 4
    mt = synth.make_model(synth.SMALL, "bf16", 2, DEV, ctx=40, steps=k)
    om = oracle_model(mt)
    dec = api.Decoder(mt, max_steps=k, verify_k=k)
    draft = [int(t) for t in np.random.default_rng(5).integers(0, mt.shape.vocab, k - 1)]
    dec.verify(torch.tensor(draft, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    _check_pass(dec, mt, om, [], draft, int(mt.seq_lens[0]), 0, ["bf16"], TOL["bf16"])
    assert api.check_device_error() == 0
