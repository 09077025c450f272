"""The allocation-free attention entry point, qd_attn_decode_paged_noalloc.

It serves callers that cannot allocate device memory (a host that reserved all
device memory for its own pool, a plugin handed only its input and output
buffers, a latency-critical loop that must not pay cudaMalloc's implicit
synchronisation): the split-KV scratch is a static 8 MiB array in the library.
Its results must match qd_attn_decode_paged with a caller-provided workspace,
call after call, and shapes whose scratch does not fit must be refused.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import rel_max_abs
from transformer_decode_step_weight_gb300 import api, synth

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = 1e-5   # the attention parity tolerance used elsewhere


def _case(seed, lens, hq=32, hkv=8, ps=16):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    B = len(lens)
    per = [max(1, -(-n // ps)) for n in lens]
    max_pages = max(per)
    n_pages = sum(per) + 2
    perm = torch.randperm(n_pages, generator=g, device=DEV).to(torch.int32)
    pt = torch.zeros((B, max_pages), dtype=torch.int32, device=DEV)
    off = 0
    for b, n in enumerate(per):
        pt[b, :n] = perm[off:off + n]
        off += n
    kp = torch.randn((n_pages, hkv, ps, 128), generator=g, device=DEV).to(torch.bfloat16)
    vp = torch.randn((n_pages, hkv, ps, 128), generator=g, device=DEV).to(torch.bfloat16)
    q = torch.randn((B, hq, 128), generator=g, device=DEV) * 0.3
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    return q, kp, vp, pt, sl


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(cuda_lib):
    scale = 1 / math.sqrt(128)
    for seed, lens in ((1, [1, 300, 4000]), (2, [129, 2048, 65])):   # two calls in a row
        q, kp, vp, pt, sl = _case(seed, lens)
        ref = api.attn_decode_paged(q, kp, vp, pt, sl, scale)
        got = api.attn_decode_paged_noalloc(q, kp, vp, pt, sl, scale)
        torch.cuda.synchronize()
        for b in range(len(lens)):
            assert rel_max_abs(got[b].cpu().numpy(), ref[b].cpu().numpy()) < TOL, (seed, b)
            assert rel_max_abs(got[b].cpu().numpy(), _oracle_attention(q, kp, vp, pt, lens, b, scale)) < TOL
    assert api.check_device_error() == 0


def _oracle_attention(q, kp, vp, pt, lens, b, scale):
    """The oracle's GQA attention of sequence b over its gathered pages."""
    n = lens[b]
    k = oracle.bf16_to_f64(oracle.gather_paged(synth.bits_u16(kp), pt[b].cpu().numpy(), n))
    v = oracle.bf16_to_f64(oracle.gather_paged(synth.bits_u16(vp), pt[b].cpu().numpy(), n))
    return oracle.gqa_attention(q[b].double().cpu().numpy(), k, v, scale)


def test_noalloc_tensor_core_form_matches_workspace_and_oracle(cuda_lib):
    # batch x kv heads at or above the SM count: the tensor-core attention runs on the
    # static scratch (its tickets cleared by the call). Two calls in a row.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B = -(-sms // 8) + 5
    scale = 1 / math.sqrt(128)
    for seed in (3, 4):
        rng = np.random.default_rng(seed)
        lens = [int(v) for v in rng.integers(1, 300, B)]
        q, kp, vp, pt, sl = _case(seed, lens)
        assert api.attn_workspace_bytes(B, 32, 8, pt.shape[1] * 16) <= 8 << 20
        ref = api.attn_decode_paged(q, kp, vp, pt, sl, scale)
        got = api.attn_decode_paged_noalloc(q, kp, vp, pt, sl, scale)
        torch.cuda.synchronize()
        for b in range(B):
            assert rel_max_abs(got[b].cpu().numpy(), ref[b].cpu().numpy()) < TOL, (seed, b)
        for b in (0, B // 2, B - 1):
            assert rel_max_abs(got[b].cpu().numpy(), _oracle_attention(q, kp, vp, pt, lens, b, scale)) < TOL
    assert api.check_device_error() == 0


def test_noalloc_refuses_shapes_beyond_its_scratch(cuda_lib):
    B, hq, hkv, ps, max_pages = 64, 32, 8, 16, 256
    need = api.attn_workspace_bytes(B, hq, hkv, ps * max_pages)
    assert need > 8 << 20
    q = torch.zeros((B, hq, 128), device=DEV)
    kp = torch.zeros((1, hkv, ps, 128), dtype=torch.bfloat16, device=DEV)
    pt = torch.zeros((B, max_pages), dtype=torch.int32, device=DEV)
    sl = torch.zeros(B, dtype=torch.int32, device=DEV)
    out = torch.empty_like(q)
    rc = api.lib().qd_attn_decode_paged_noalloc(q.data_ptr(), kp.data_ptr(), kp.data_ptr(), pt.data_ptr(),
                                                sl.data_ptr(), B, hq, hkv, 128, ps, max_pages, 1, 0.1,
                                                out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == -4
    assert b"static array" in api.lib().qd_last_error()
    np.testing.assert_array_equal(out.shape, q.shape)
