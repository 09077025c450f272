"""Test-side glue: host copies of the seeded tensors in the oracle's form."""
from __future__ import annotations

import numpy as np

import oracle
from transformer_decode_step_weight_gb300 import synth


def oracle_dims(s: synth.Shape) -> oracle.Dims:
    return oracle.Dims(s.hidden, s.n_q_heads, s.n_kv_heads, s.head_dim, s.ffn,
                       s.rms_eps, s.rope_theta)


def oracle_layer(lt: synth.LayerTensors, wtype: str) -> oracle.LayerWeights:
    if wtype == "bf16":
        w = {k: synth.bits_u16(getattr(lt, k)) for k in ("w_qkv", "w_o", "w_gu", "w_down")}
        s = {}
    else:
        w = {k: synth.host_i8(getattr(lt, k)) for k in ("w_qkv", "w_o", "w_gu", "w_down")}
        s = {k: synth.bits_u16(getattr(lt, k)) for k in ("s_qkv", "s_o", "s_gu", "s_down")}
    n = {k: synth.bits_u16(getattr(lt, k)) for k in ("ln_in", "ln_post", "q_norm", "k_norm")}
    return oracle.LayerWeights(**w, **n, **s)


def oracle_model(mt: synth.ModelTensors) -> oracle.Model:
    layers = [oracle_layer(lt, mt.wtype) for lt in mt.layers]
    if mt.lm_head_scales is not None:
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
