"""Test-side glue: host copies of the seeded tensors in the oracle's form, and the
teacher-forced comparison of a GPU decode run with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from transformer_decode_step_weight_gb300 import synth


def oracle_dims(s: synth.Shape) -> oracle.Dims:
    return oracle.Dims(s.hidden, s.n_q_heads, s.n_kv_heads, s.head_dim, s.ffn,
                       s.rms_eps, s.rope_theta)


def oracle_layer(lt: synth.LayerTensors, wtype: str) -> oracle.LayerWeights:
    if wtype == "bf16":
        w = {k: synth.bits_u16(getattr(lt, k)) for k in ("w_qkv", "w_o", "w_gu", "w_down")}
        s = {}
    elif wtype == "int4":
        w = {k: synth.host_u8(getattr(lt, k)) for k in ("w_qkv", "w_o", "w_gu", "w_down")}
        s = {k: synth.bits_u16(getattr(lt, k)) for k in ("s_qkv", "s_o", "s_gu", "s_down")}
    else:
        w = {k: synth.host_i8(getattr(lt, k)) for k in ("w_qkv", "w_o", "w_gu", "w_down")}
        s = {k: synth.bits_u16(getattr(lt, k)) for k in ("s_qkv", "s_o", "s_gu", "s_down")}
    n = {k: synth.bits_u16(getattr(lt, k)) for k in ("ln_in", "ln_post", "q_norm", "k_norm")}
    return oracle.LayerWeights(**w, **n, **s)


def oracle_model(mt: synth.ModelTensors) -> oracle.Model:
    layers = [oracle_layer(lt, mt.wtype) for lt in mt.layers]
    if mt.lm_head_scales is not None and mt.lm_head.dtype == torch.uint8:
        lm, lms = synth.host_u8(mt.lm_head), synth.bits_u16(mt.lm_head_scales)
    elif mt.lm_head_scales is not None:
        lm, lms = synth.host_i8(mt.lm_head), synth.bits_u16(mt.lm_head_scales)
    else:
        lm, lms = synth.bits_u16(mt.lm_head), None
    return oracle.Model(oracle_dims(mt.shape), layers, synth.bits_u16(mt.embed),
                        synth.bits_u16(mt.final_norm), lm, lms)


def oracle_caches(mt: synth.ModelTensors, b: int, n_tokens: int):
    """Logical float64 [Hkv, n_tokens, D] caches of sequence b, one per layer,
    with room for ``n_tokens`` (slots past the cached length are zero)."""
    pt = mt.page_table[b].cpu().numpy()
    ks, vs = [], []
    have = int(mt.seq_lens[b])
    for kc, vc in zip(mt.k_cache, mt.v_cache):
        k = oracle.bf16_to_f64(oracle.gather_paged(synth.bits_u16(kc), pt, have))
        v = oracle.bf16_to_f64(oracle.gather_paged(synth.bits_u16(vc), pt, have))
        K = np.zeros((k.shape[0], n_tokens, k.shape[2]))
        V = np.zeros_like(K)
        K[:, :have] = k
        V[:, :have] = v
        ks.append(K)
        vs.append(V)
    return ks, vs


def rel_max_abs(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-300))


# Relative max-abs error limits on logits / hidden states: BF16 path, f32-activation
# Q8_0 lane, dp4a lane, and the batched Q8_0 path (tensor cores, weights widened).
TOL = {"bf16": 2e-2, "f32": 5e-3, "i8": 2e-2, "w_bf16": 2e-2}


def teacher_forced(dec, mt, steps, lanes, b=0, floor_factor=None, lm_resync=False):
    """Run `steps` eager GPU decode steps of sequence b; check each against the oracle.

    Protocol for greedy tokens (teacher-forced): the oracle follows the GPU's own
    token stream. ``lanes`` is a list of (mode, act, lm_act, tol) oracle lanes the GPU
    logits are held to, each with its own caches. At every step the logits must be
    within the lane's relative max-abs tolerance, the GPU token must be the argmax of
    the GPU logits, and it must equal the oracle's argmax unless the oracle's top-1 /
    top-2 gap is below 4x the step's max-abs logit error (a near tie, logged). The
    first lane decides the token agreement figures.

    floor_factor: the end-to-end limit of lane 0 at each step becomes max(tol,
    floor_factor x the oracle's own drift at that step), the drift being how far the
    oracle's logits move when its sums are accumulated in binary32 instead of float64
    (``acc="f32"``, a second oracle run on its own caches, teacher-forced on the same
    tokens). In a deep model of bf16-rounded activations, ulp-level differences flip
    roundings that the following layers amplify; this measures that floor for the
    model at hand.
    lm_resync: at step 0 also hold the GPU logits to the oracle's LM head applied to
    the GPU's own final hidden state (every row), at the lane's tolerance.
    Returns the log dict.
    """
    import torch

    from transformer_decode_step_weight_gb300 import api
    import oracle

    om = oracle_model(mt)
    pos0 = int(mt.seq_lens[b])
    caches = [oracle_caches(mt, b, pos0 + steps) for _ in lanes]
    caches32 = oracle_caches(mt, b, pos0 + steps) if floor_factor is not None else None
    tok = int(mt.start_tok[b])
    tols = [ln[3] for ln in lanes]
    st = {"steps": steps, "strict": 0, "near_ties": [], "worst_rel_err": [0.0] * len(lanes),
          "lanes": [f"{m}/{a}/{la or a}" for m, a, la, _ in lanes], "floor": [], "tol": []}
    for t in range(steps):
        dec.step()
        torch.cuda.synchronize()
        g = dec.logits[b].double().cpu().numpy()
        gtok = int(dec.tok[b])
        assert gtok == oracle.argmax_first(g), t
        assert int(dec.out_tokens[b, t]) == gtok
        for li, (mode, act, lm_act, tol) in enumerate(lanes):
            ref = oracle.decode_token(om, tok, pos0 + t, caches[li][0], caches[li][1], mode=mode, act=act,
                                      lm_act=lm_act)
            if li == 0 and floor_factor is not None:
                r32 = oracle.decode_token(om, tok, pos0 + t, caches32[0], caches32[1], mode=mode, act=act,
                                          lm_act=lm_act, acc="f32")
                fl = rel_max_abs(r32, ref)
                st["floor"].append(fl)
                tols[0] = max(tol, floor_factor * fl)
                st["tol"].append(tols[0])
            if t == 0 and li == 0 and lm_resync:
                xf = oracle.rmsnorm(dec.residual()[b].double().cpu().numpy(), oracle.bf16_to_f64(om.final_norm),
                                    om.dims.rms_eps, mode)
                lm_ref = oracle.project(om.lm_head, om.lm_head_scales, xf, lm_act or act)
                st["lm_head_resync_err"] = rel_max_abs(g, lm_ref)
                assert st["lm_head_resync_err"] < lanes[0][3], st["lm_head_resync_err"]
            err = rel_max_abs(g, ref)
            st["worst_rel_err"][li] = max(st["worst_rel_err"][li], err)
            assert err < tols[li], (t, li, err, tols[li])
            otok = oracle.argmax_first(ref)
            if gtok != otok:
                top = np.sort(ref)[-2:]
                gap = float(top[1] - top[0])
                assert gap < 4 * np.max(np.abs(g - ref)), (t, li, gtok, otok, gap)
                if li == 0:
                    st["near_ties"].append({"step": t, "gpu": gtok, "oracle": otok, "gap": gap})
            elif li == 0:
                st["strict"] += 1
        tok = gtok
    assert api.check_device_error() == 0
    return st


def per_layer_resync(mt, lane, mode, act, tol, b=0):
    """Step 0 of a contiguous-cache model one layer at a time, on the GPU's own inputs.

    The GPU's residual after l layers comes from a decoder over the first l layers of
    the same tensors (the step is deterministic, so layer l - 1 sees the same input
    inside every prefix); the oracle applies layer l - 1 to the GPU's residual after
    l - 1 layers. Each layer's output and the K/V row it writes to the cache are held
    to `tol`, so rounding differences do not compound across layers here. Returns the
    worst error of each.
    """
    import dataclasses

    import torch

    from transformer_decode_step_weight_gb300 import api
    import oracle

    om = oracle_model(mt)
    pos = int(mt.seq_lens[b])
    ks, vs = oracle_caches(mt, b, pos + 1)
    x = oracle.bf16_to_f64(synth.bits_u16(mt.embed[int(mt.start_tok[b])]))
    worst = {"layer": 0.0, "kv": 0.0}
    for li in range(len(mt.layers)):
        sub = dataclasses.replace(mt, layers=mt.layers[:li + 1], k_cache=mt.k_cache[:li + 1],
                                  v_cache=mt.v_cache[:li + 1])
        dec = api.Decoder(sub, max_steps=1, act=lane)
        dec.step()
        torch.cuda.synchronize()
        got = dec.residual()[b].double().cpu().numpy()
        dec.close()
        ref = oracle.layer_step(om.dims, om.layers[li], x, ks[li], vs[li], pos, mode=mode, act=act)
        err = rel_max_abs(got, ref)
        worst["layer"] = max(worst["layer"], err)
        assert err < tol, (li, err)
        page = int(mt.page_table[b, pos // mt.page_size])
        slot = pos % mt.page_size
        for cache, ref_c in ((mt.k_cache[li], ks[li]), (mt.v_cache[li], vs[li])):
            row = oracle.bf16_to_f64(synth.bits_u16(cache[page, :, slot, :]))
            e = rel_max_abs(row, ref_c[:, pos])
            worst["kv"] = max(worst["kv"], e)
            assert e < tol, (li, e)
        x = got
    return worst
