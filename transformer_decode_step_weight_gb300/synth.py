"""Seeded synthetic inputs for the decode step (weights, KV cache, tokens).

This module only draws random numbers and lays them out; it holds none of the
decode arithmetic. Both the CUDA library (through the tests and the bench) and
the CPU oracle receive the tensors it makes, so it is the one piece of code the
two sides share.

Distributions (the workloads the decode step is measured on): projection
weights ~ N(0, 0.02) in bf16; norm weights 1 + N(0, 0.1) in bf16; input hidden
~ N(0, 1); KV cache ~ N(0, 1) in bf16; Q8_0 weights are integers uniform in
[-127, 127] with fp16 scales |N(0, 0.002)|; the start token is uniform in
[0, vocab). Draw order for a model, from one ``torch.Generator`` seeded once:
embedding; per layer (w_qkv, w_o, w_gu, w_down, ln_in, ln_post, q_norm,
k_norm), each Q8_0 matrix drawing its int8 values then its scales; final norm;
LM head (untied models only); per layer K cache then V cache; start token.

Storage layouts:
  * bf16 weights: row-major [rows, cols]; w_qkv rows = [q (Hq*D); k (Hkv*D);
    v (Hkv*D)], w_gu rows = [gate (F); up (F)].
  * Q8_0 weights: int8 values [rows, cols] and fp16 scales [rows, cols/32],
    two separate row-major arrays.
  * INT4 weights: packed uint8 [rows, cols/2] (two offset-binary nibbles q + 8 per
    byte, the even column in the low nibble) and fp16 per-row scales [rows].
  * KV cache: bf16 [pages, Hkv, page_size, D]; a contiguous cache is one page of
    ``max_ctx`` tokens per sequence.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Shape:
    name: str
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    n_layers: int
    vocab: int
    tied: bool
    rms_eps: float = 1e-6
    rope_theta: float = 1e6

    @property
    def qkv_rows(self):
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim


QWEN3_06B = Shape("qwen3-0.6b", 1024, 16, 8, 128, 3072, 28, 151936, True)
QWEN3_8B = Shape("qwen3-8b", 4096, 32, 8, 128, 12288, 36, 151936, False)
# small shapes for fast parity cases (several tiles, ragged tails)
TINY = Shape("tiny", 256, 4, 2, 128, 544, 2, 1000, True)
SMALL = Shape("small", 512, 8, 2, 128, 1376, 3, 5003, False)
# dims that are multiples of 64, as the batched (tensor-core) projections need
SMALL64 = Shape("small64", 512, 8, 2, 128, 1408, 2, 2999, False)
# dims that are multiples of 256, as the batched Q8_0 projections need
SMALL256 = Shape("small256", 512, 4, 2, 128, 1536, 2, 3001, False)
# an INT4 parity shape: several CTA row spans, K per row a few 32-column chunks
SMALL_W4 = Shape("small_w4", 768, 4, 2, 128, 2080, 3, 4099, False)


@dataclass
class Workload:
    """One benchmark / parity workload: a shape plus context and batch."""
    name: str
    shape: Shape
    wtype: str          # "bf16" | "q8_0"
    ctx: int            # tokens already in the cache before the first step
    steps: int          # decode steps
    batch: int = 1
    paged: bool = False
    page_size: int = 16
    n_layers: int | None = None   # override (single-layer workload)
    description: str = ""

    @property
    def layers(self):
        return self.shape.n_layers if self.n_layers is None else self.n_layers


WORKLOADS = {
    "qwen3-0.6b-layer": Workload(
        "qwen3-0.6b-layer", QWEN3_06B, "bf16", ctx=128, steps=1, n_layers=1,
        description="one Qwen3-0.6B-shaped decoder layer, one decode step at position 128"),
    "qwen3-0.6b": Workload(
        "qwen3-0.6b", QWEN3_06B, "bf16", ctx=2048, steps=128,
        description="Qwen3-0.6B-shaped model, tied LM head, contiguous KV at context 2048"),
    "qwen3-8b-bf16": Workload(
        "qwen3-8b-bf16", QWEN3_8B, "bf16", ctx=4096, steps=128,
        description="Qwen3-8B-shaped BF16 model, batch 1, KV at context 4096, 128 greedy steps"),
    "qwen3-8b-int4": Workload(
        "qwen3-8b-int4", QWEN3_8B, "int4", ctx=4096, steps=128,
        description="Qwen3-8B-shaped W4A16 model (INT4 per-row-scaled weights, LM head INT4 too), batch 1, "
                    "context 4096"),
    "qwen3-8b-q8_0": Workload(
        "qwen3-8b-q8_0", QWEN3_8B, "q8_0", ctx=2048, steps=128,
        description="Qwen3-8B-shaped Q8_0 model (LM head Q8_0 too), batch 1, context 2048"),
    **{f"qwen3-8b-bf16-b{n}": Workload(
        f"qwen3-8b-bf16-b{n}", QWEN3_8B, "bf16", ctx=2048, steps=128, batch=n,
        description=f"Qwen3-8B-shaped BF16 model, {n} sequences, contiguous KV at context 2048 each")
       for n in (2, 4, 8)},
    "qwen3-8b-bf16-paged-b64": Workload(
        "qwen3-8b-bf16-paged-b64", QWEN3_8B, "bf16", ctx=4096, steps=64, batch=64, paged=True,
        description="64 sequences, context uniform in [128, 4096], 16-token pages, random page table"),
    "qwen3-8b-q8_0-paged-b64": Workload(
        "qwen3-8b-q8_0-paged-b64", QWEN3_8B, "q8_0", ctx=4096, steps=64, batch=64, paged=True,
        description="Q8_0 weights (LM head too), 64 sequences, context uniform in [128, 4096], 16-token pages"),
}


def _normal_bf16(gen, shape, std, device, mean=0.0):
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(torch.bfloat16)


def _int4(gen, rows, cols, device):
    """INT4 weights: codes uniform in [-8, 7] packed two per byte as offset-binary
    nibbles (even column low), fp16 per-row scales |N(0, 0.01)|."""
    q = torch.randint(0, 16, (rows, cols), generator=gen, device=device, dtype=torch.int16)
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).to(torch.uint8)
    d = torch.randn((rows,), generator=gen, device=device, dtype=torch.float32).abs_().mul_(0.01).to(torch.float16)
    return packed, d


def _q8_0(gen, rows, cols, device):
    qs = torch.randint(-127, 128, (rows, cols), generator=gen, device=device,
                       dtype=torch.int16).to(torch.int8)
    d = torch.randn((rows, cols // 32), generator=gen, device=device, dtype=torch.float32)
    d = d.abs_().mul_(0.002).to(torch.float16)
    return qs, d


@dataclass
class LayerTensors:
    w_qkv: torch.Tensor
    w_o: torch.Tensor
    w_gu: torch.Tensor
    w_down: torch.Tensor
    ln_in: torch.Tensor
    ln_post: torch.Tensor
    q_norm: torch.Tensor
    k_norm: torch.Tensor
    s_qkv: torch.Tensor | None = None
    s_o: torch.Tensor | None = None
    s_gu: torch.Tensor | None = None
    s_down: torch.Tensor | None = None


def make_layer(gen, s: Shape, wtype: str, device) -> LayerTensors:
    mats = {"w_qkv": (s.qkv_rows, s.hidden), "w_o": (s.hidden, s.n_q_heads * s.head_dim),
            "w_gu": (2 * s.ffn, s.hidden), "w_down": (s.hidden, s.ffn)}
    out = {}
    for k, (r, c) in mats.items():
        if wtype == "bf16":
            out[k] = _normal_bf16(gen, (r, c), 0.02, device)
        elif wtype == "q8_0":
            out[k], out["s" + k[1:]] = _q8_0(gen, r, c, device)
        elif wtype == "int4":
            out[k], out["s" + k[1:]] = _int4(gen, r, c, device)
        else:
            raise ValueError(wtype)
    out["ln_in"] = _normal_bf16(gen, (s.hidden,), 0.1, device, mean=1.0)
    out["ln_post"] = _normal_bf16(gen, (s.hidden,), 0.1, device, mean=1.0)
    out["q_norm"] = _normal_bf16(gen, (s.head_dim,), 0.1, device, mean=1.0)
    out["k_norm"] = _normal_bf16(gen, (s.head_dim,), 0.1, device, mean=1.0)
    return LayerTensors(**out)


@dataclass
class ModelTensors:
    shape: Shape
    wtype: str
    layers: list
    embed: torch.Tensor
    final_norm: torch.Tensor
    lm_head: torch.Tensor
    lm_head_scales: torch.Tensor | None
    k_cache: list = field(default_factory=list)   # per layer [pages, Hkv, ps, D]
    v_cache: list = field(default_factory=list)
    page_table: torch.Tensor | None = None        # int32 [B, max_pages]
    seq_lens: torch.Tensor | None = None          # int32 [B] tokens already cached
    page_size: int = 0
    max_pages: int = 0
    start_tok: torch.Tensor | None = None         # int32 [B]


def make_model(s: Shape, wtype: str, seed: int, device, *, n_layers: int | None = None,
               batch: int = 1, ctx: int | list = 0, steps: int = 1, paged: bool = False,
               page_size: int = 16, lm_wtype: str | None = None) -> ModelTensors:
    """Seeded random-init model plus a KV cache holding ``ctx`` tokens per sequence.

    Contiguous cache (paged=False): one page of ``max_ctx = max(ctx) + steps``
    tokens per sequence, page table [[0], [1], ...]. Paged cache: each sequence
    gets ceil((ctx_b + steps) / page_size) pages drawn from a seeded random
    permutation of all physical pages.
    ``ctx`` may be an int (all sequences) or a list of per-sequence lengths; for
    the paged workload pass ``ctx=None`` to draw lengths uniform in [128, 4096].
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    L = s.n_layers if n_layers is None else n_layers
    lm_wtype = wtype if lm_wtype is None else lm_wtype
    embed = _normal_bf16(gen, (s.vocab, s.hidden), 0.02, device)
    layers = [make_layer(gen, s, wtype, device) for _ in range(L)]
    final_norm = _normal_bf16(gen, (s.hidden,), 0.1, device, mean=1.0)
    lm_scales = None
    if lm_wtype == "q8_0":
        lm_head, lm_scales = _q8_0(gen, s.vocab, s.hidden, device)
    elif lm_wtype == "int4":
        lm_head, lm_scales = _int4(gen, s.vocab, s.hidden, device)
    elif s.tied:
        lm_head = embed
    else:
        lm_head = _normal_bf16(gen, (s.vocab, s.hidden), 0.02, device)

    if ctx is None:
        lens = torch.randint(128, 4097, (batch,), generator=gen, device=device,
                             dtype=torch.int64).to(torch.int32)
    elif isinstance(ctx, int):
        lens = torch.full((batch,), ctx, dtype=torch.int32, device=device)
    else:
        lens = torch.tensor(list(ctx), dtype=torch.int32, device=device)
    lens_h = [int(v) for v in lens.cpu()]
    if paged:
        per_seq = [-(-(n + steps) // page_size) for n in lens_h]
        max_pages = max(per_seq)
        n_phys = sum(per_seq)
        perm = torch.randperm(n_phys, generator=gen, device=device).to(torch.int32)
        pt = torch.zeros((batch, max_pages), dtype=torch.int32, device=device)
        off = 0
        for b, n in enumerate(per_seq):
            pt[b, :n] = perm[off:off + n]
            off += n
        ps = page_size
    else:
        max_ctx = max(lens_h) + steps
        n_phys, max_pages, ps = batch, 1, max_ctx
        pt = torch.arange(batch, dtype=torch.int32, device=device).reshape(batch, 1)
    kc, vc = [], []
    for _ in range(L):
        kc.append(_normal_bf16(gen, (n_phys, s.n_kv_heads, ps, s.head_dim), 1.0, device))
        vc.append(_normal_bf16(gen, (n_phys, s.n_kv_heads, ps, s.head_dim), 1.0, device))
    start = torch.randint(0, s.vocab, (batch,), generator=gen, device=device,
                          dtype=torch.int64).to(torch.int32)
    return ModelTensors(s, wtype, layers, embed, final_norm, lm_head, lm_scales, kc, vc,
                        pt, lens, ps, max_pages, start)


def make_hidden(seed: int, n: int, device, batch: int = 1) -> torch.Tensor:
    """Input hidden state ~ N(0, 1), float32 [batch, n] (single-layer workload)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return torch.randn((batch, n), generator=gen, device=device, dtype=torch.float32)


# --------------------------------------------------------------------------
# host copies for the oracle (bit-exact views; no arithmetic)
# --------------------------------------------------------------------------


def bits_u16(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit storage (bf16 or fp16) as a host uint16 array."""
    assert t.element_size() == 2
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_i8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().astype(np.int8)


def host_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().astype(np.uint8)
