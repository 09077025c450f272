"""Thin ctypes binding of libqd.so (argument marshalling only).

Every function here forwards device pointers (``tensor.data_ptr()``), sizes
and the current CUDA stream to the C ABI declared in ``include/qd.h``; all
arithmetic of the decode step runs in the library's CUDA kernels. PyTorch only
allocates device memory and supplies streams. If the library has not been
built, the first call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqd.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "qd.h")

QD_OK = 0
QD_W_BF16, QD_W_Q8_0, QD_W_INT4 = 0, 1, 2
QD_ACT_F32, QD_ACT_I8 = 0, 1
DEVERR = {1: "page", 2: "pos", 4: "nan", 8: "steps", 16: "timeout"}

_vp = C.c_void_p
_i = C.c_int
_f = C.c_float
_sz = C.c_size_t


class LayerDims(C.Structure):
    _fields_ = [("hidden", _i), ("n_q_heads", _i), ("n_kv_heads", _i), ("head_dim", _i), ("ffn", _i),
                ("rms_eps", _f), ("rope_theta", _f), ("wtype", _i), ("act", _i)]


class LayerWeights(C.Structure):
    _fields_ = [(n, _vp) for n in ("w_qkv", "w_o", "w_gu", "w_down", "s_qkv", "s_o", "s_gu", "s_down",
                                   "ln_in", "ln_post", "q_norm", "k_norm")]


class StepArgs(C.Structure):
    _fields_ = [("layers", _vp), ("n_layers", _i),
                ("embed", _vp), ("final_norm", _vp), ("lm_head", _vp), ("lm_head_scales", _vp),
                ("lm_act", _i), ("vocab", _i),
                ("k_cache", _vp), ("v_cache", _vp),
                ("page_table", _vp), ("page_size", _i), ("max_pages", _i), ("n_pages", _i),
                ("rope_table", _vp), ("rope_max_pos", _i),
                ("tok", _vp), ("pos", _vp), ("step", _vp), ("out_tokens", _vp),
                ("max_steps", _i), ("batch", _i),
                ("logits", _vp), ("workspace", _vp), ("workspace_bytes", _sz),
                ("lm_wtype", _i), ("top_k", _i), ("topk_ids", _vp), ("topk_vals", _vp)]


_SIGS = {
    "qd_last_error": (C.c_char_p, []),
    "qd_version": (_i, []),
    "qd_gemv_bf16": (_i, [_vp, _i, _i, _vp, _i, _vp, _i, _vp]),
    "qd_gemv_q8_0": (_i, [_vp, _vp, _i, _i, _vp, _vp, _vp, _i, _vp, _vp]),
    "qd_quantize_q8_0": (_i, [_vp, _i, _vp, _vp, _vp]),
    "qd_gemv_w4": (_i, [_vp, _vp, _i, _i, _vp, _vp, _vp]),
    "qd_w4_topk_workspace_bytes": (_sz, []),
    "qd_gemv_w4_topk": (_i, [_vp, _vp, _i, _i, _vp, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
    "qd_gemm_workspace_bytes": (_sz, [_i, _i, _i]),
    "qd_gemm_q8_0": (_i, [_vp, _vp, _i, _i, _vp, _i, _vp, _vp, _sz, _vp]),
    "qd_attn_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "qd_attn_decode_paged": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _vp, _sz, _vp]),
    "qd_attn_decode_paged_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _vp]),
    "qd_argmax_workspace_bytes": (_sz, [_i]),
    "qd_argmax_advance": (_i, [_vp, _i, _i, _vp, _vp, _vp, _vp, _i, _vp, _sz, _vp]),
    "qd_rope_table_init": (_i, [_vp, _i, _i, _f, _vp]),
    "qd_create_layer": (_i, [C.POINTER(LayerDims), C.POINTER(LayerWeights), C.POINTER(_vp)]),
    "qd_destroy_layer": (_i, [_vp]),
    "qd_step_workspace_bytes": (_sz, [C.POINTER(StepArgs)]),
    "qd_decode_step": (_i, [C.POINTER(StepArgs), _vp]),
    "qd_step_launch_count": (_i, [C.POINTER(StepArgs)]),
    "qd_graph_create": (_i, [C.POINTER(StepArgs), _i, _vp, C.POINTER(_vp)]),
    "qd_graph_launch": (_i, [_vp, _vp]),
    "qd_graph_destroy": (_i, [_vp]),
    "qd_check_device_error": (_i, [_vp, C.POINTER(_i)]),
    "qd_verify_workspace_bytes": (_sz, [C.POINTER(StepArgs), _i]),
    "qd_verify_step": (_i, [C.POINTER(StepArgs), _vp, _i, _vp, _vp, _vp, _vp]),
    "qd_prefill_workspace_bytes": (_sz, [C.POINTER(StepArgs), _i]),
    "qd_prefill": (_i, [C.POINTER(StepArgs), _vp, _i, _vp, _vp]),
    "qd_debug_wait_timeout": (_i, [_i, _vp]),
    "qd_gemv_w4_workspace_bytes": (_sz, [_i, _i]),
    "qd_gemv_w4_ex": (_i, [_vp, _vp, _i, _i, _vp, _vp, _vp, _sz, _vp]),
    "qd_debug_q8_block_dots": (_i, [_vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp]),
    "qd_debug_paged_indices": (_i, [_vp, _i, _i, _i, _i, _i, _vp, _vp]),
}

_lib = None


def lib():
    """Load libqd.so once; raise if it is missing (no CPU fallback exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run transformer_decode_step_weight_gb300.build")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/qd.h declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qd_[a-z0-9_]+)\s*\(", src)))


class QDError(RuntimeError):
    pass


def _check(rc: int):
    if rc != QD_OK:
        raise QDError(f"libqd error {rc}: {lib().qd_last_error().decode()}")


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _p(t):
    return None if t is None else t.data_ptr()


# ---------------------------------------------------------------- single ops


def gemv_bf16(W, x, y=None, stream=None):
    """y[b] = W @ x[b]; W bf16 [R, K]; x bf16 or f32 [B, K] -> f32 [B, R]."""
    x2 = x if x.dim() == 2 else x.reshape(1, -1)
    R, K = W.shape
    if y is None:
        y = torch.empty((x2.shape[0], R), dtype=torch.float32, device=W.device)
    _check(lib().qd_gemv_bf16(_p(W), R, K, _p(x2), int(x2.dtype == torch.float32), _p(y), x2.shape[0],
                              _stream(stream)))
    return y


def gemv_q8_0(qs, d, x=None, xq=None, xd=None, act=QD_ACT_F32, y=None, stream=None):
    R, K = qs.shape
    if y is None:
        y = torch.empty(R, dtype=torch.float32, device=qs.device)
    _check(lib().qd_gemv_q8_0(_p(qs), _p(d), R, K, _p(x), _p(xq), _p(xd), act, _p(y), _stream(stream)))
    return y


def debug_wait_timeout(limit_us: int, stream=None):
    """Run a bounded wait that nothing completes (QD_DEVERR_TIMEOUT afterwards)."""
    _check(lib().qd_debug_wait_timeout(int(limit_us), _stream(stream)))


def gemv_w4_workspace_bytes(R: int, K: int) -> int:
    return int(lib().qd_gemv_w4_workspace_bytes(R, K))


def gemv_w4(W, d, x, y=None, workspace=None, stream=None):
    """y = (d * q) @ x; W packed uint8 [R, K / 2], d f16 [R], x bf16 [K] -> f32 [R].
    `workspace` (zero-filled uint8, gemv_w4_workspace_bytes) lets small matrices split K."""
    R, Kh = W.shape
    if y is None:
        y = torch.empty(R, dtype=torch.float32, device=W.device)
    if workspace is None:
        _check(lib().qd_gemv_w4(_p(W), _p(d), R, 2 * Kh, _p(x), _p(y), _stream(stream)))
    else:
        _check(lib().qd_gemv_w4_ex(_p(W), _p(d), R, 2 * Kh, _p(x), _p(y), _p(workspace), workspace.numel(),
                                   _stream(stream)))
    return y


def gemv_w4_topk(W, d, x, k, y=None, workspace=None, stream=None):
    """(logits, top-k ids, top-k values) of the INT4 LM-head form."""
    R, Kh = W.shape
    if y is None:
        y = torch.empty(R, dtype=torch.float32, device=W.device)
    if workspace is None:
        workspace = torch.zeros(int(lib().qd_w4_topk_workspace_bytes()), dtype=torch.uint8, device=W.device)
    ids = torch.empty(k, dtype=torch.int32, device=W.device)
    vals = torch.empty(k, dtype=torch.float32, device=W.device)
    _check(lib().qd_gemv_w4_topk(_p(W), _p(d), R, 2 * Kh, _p(x), k, _p(y), _p(ids), _p(vals), _p(workspace),
                                 workspace.numel(), _stream(stream)))
    return y, ids, vals


def gemm_workspace_bytes(rows, cols, wtype=QD_W_Q8_0):
    return int(lib().qd_gemm_workspace_bytes(rows, cols, wtype))


def gemm_q8_0(qs, d, x, y=None, workspace=None, stream=None):
    """y[b] = bf16(f32(d) * qs) @ x[b] on the tensor cores; x bf16 [B, K] -> f32 [B, R]."""
    R, K = qs.shape
    B = x.shape[0]
    if y is None:
        y = torch.empty((B, R), dtype=torch.float32, device=qs.device)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().qd_gemm_q8_0(_p(qs), _p(d), R, K, _p(x), B, _p(y), _p(workspace), nbytes, _stream(stream)))
    return y


def quantize_q8_0(x, stream=None):
    n = x.numel()
    xq = torch.empty(n, dtype=torch.int8, device=x.device)
    xd = torch.empty(n // 32, dtype=torch.float16, device=x.device)
    _check(lib().qd_quantize_q8_0(_p(x), n, _p(xq), _p(xd), _stream(stream)))
    return xq, xd


def attn_workspace_bytes(batch, hq, hkv, max_ctx):
    return int(lib().qd_attn_workspace_bytes(batch, hq, hkv, max_ctx))


def attn_decode_paged(q, k_pages, v_pages, page_table, seq_lens, scale, out=None, workspace=None, stream=None):
    """q f32 [B, Hq, D]; caches bf16 [n_pages, Hkv, ps, D]; page_table int32 [B, max_pages]."""
    B, Hq, D = q.shape
    n_pages, Hkv, ps, _ = k_pages.shape
    max_pages = page_table.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = torch.zeros(attn_workspace_bytes(B, Hq, Hkv, max_pages * ps), dtype=torch.uint8,
                                device=q.device)
    _check(lib().qd_attn_decode_paged(_p(q), _p(k_pages), _p(v_pages), _p(page_table), _p(seq_lens), B, Hq, Hkv,
                                      D, ps, max_pages, n_pages, float(scale), _p(out), _p(workspace),
                                      workspace.numel(), _stream(stream)))
    return out


def attn_decode_paged_noalloc(q, k_pages, v_pages, page_table, seq_lens, scale, out=None, stream=None):
    """qd_attn_decode_paged with the library's static scratch instead of a workspace."""
    B, Hq, D = q.shape
    n_pages, Hkv, ps, _ = k_pages.shape
    if out is None:
        out = torch.empty_like(q)
    _check(lib().qd_attn_decode_paged_noalloc(_p(q), _p(k_pages), _p(v_pages), _p(page_table), _p(seq_lens), B,
                                              Hq, Hkv, D, ps, page_table.shape[1], n_pages, float(scale), _p(out),
                                              _stream(stream)))
    return out


def argmax_advance(logits, tok, pos, step, out_tokens, workspace=None, stream=None):
    B, V = logits.shape
    if workspace is None:
        workspace = torch.zeros(int(lib().qd_argmax_workspace_bytes(B)), dtype=torch.uint8, device=logits.device)
    _check(lib().qd_argmax_advance(_p(logits), V, B, _p(tok), _p(pos), _p(step), _p(out_tokens),
                                   out_tokens.shape[1], _p(workspace), workspace.numel(), _stream(stream)))


def rope_table(max_pos, head_dim, theta, device, stream=None):
    t = torch.empty((max_pos, head_dim // 2, 2), dtype=torch.float32, device=device)
    _check(lib().qd_rope_table_init(_p(t), max_pos, head_dim, float(theta), _stream(stream)))
    return t


def check_device_error(stream=None) -> int:
    bits = _i(0)
    _check(lib().qd_check_device_error(_stream(stream), C.byref(bits)))
    return bits.value


def debug_q8_block_dots(qs, d, xq, xd, stream=None):
    """(int32 block dots [R, K/32], f32 y [R]) of the production i8-lane Q8_0 GEMV."""
    R, K = qs.shape
    dots = torch.empty((R, K // 32), dtype=torch.int32, device=qs.device)
    y = torch.empty(R, dtype=torch.float32, device=qs.device)
    _check(lib().qd_debug_q8_block_dots(_p(qs), _p(d), R, K, _p(xq), _p(xd), _p(dots), _p(y), _stream(stream)))
    return dots, y


def debug_paged_indices(page_table, page_size, n_tokens, n_pages=None, stream=None):
    B, max_pages = page_table.shape
    if n_pages is None:
        n_pages = max_pages * B
    idx = torch.empty((B, n_tokens), dtype=torch.int32, device=page_table.device)
    _check(lib().qd_debug_paged_indices(_p(page_table), B, max_pages, page_size, n_pages, n_tokens, _p(idx),
                                        _stream(stream)))
    return idx


# ---------------------------------------------------------------- whole step


class Decoder:
    """Owns the layer handles, step state and workspace of one decode run.

    ``model`` holds device tensors (see ``synth.ModelTensors``): per-layer
    weights, embedding, final norm, LM head, the per-layer K/V caches, page
    table, cached lengths and start tokens. The state buffers (tok, pos, step,
    out_tokens) are device int32 tensors advanced by the library.
    """

    def __init__(self, model, max_steps: int, act: int = QD_ACT_F32, lm_act: int | None = None,
                 device="cuda", verify_k: int = 0, top_k: int = 0, prefill_max: int = 0):
        self.m = model
        s = model.shape
        self.device = torch.device(device)
        wt = {"bf16": QD_W_BF16, "q8_0": QD_W_Q8_0, "int4": QD_W_INT4}[model.wtype]
        dims = LayerDims(s.hidden, s.n_q_heads, s.n_kv_heads, s.head_dim, s.ffn, s.rms_eps, s.rope_theta,
                         wt, act)
        self._handles = []
        for lt in model.layers:
            w = LayerWeights(_p(lt.w_qkv), _p(lt.w_o), _p(lt.w_gu), _p(lt.w_down),
                             _p(lt.s_qkv), _p(lt.s_o), _p(lt.s_gu), _p(lt.s_down),
                             _p(lt.ln_in), _p(lt.ln_post), _p(lt.q_norm), _p(lt.k_norm))
            h = _vp()
            _check(lib().qd_create_layer(C.byref(dims), C.byref(w), C.byref(h)))
            self._handles.append(h)
        L = len(self._handles)
        self._layer_arr = (_vp * L)(*[h.value for h in self._handles])
        self._k_arr = (_vp * L)(*[_p(t) for t in model.k_cache])
        self._v_arr = (_vp * L)(*[_p(t) for t in model.v_cache])
        B = int(model.start_tok.numel())
        self.batch = B
        self.max_steps = max_steps
        self.tok = model.start_tok.clone().to(torch.int32)
        self.pos = model.seq_lens.clone().to(torch.int32)
        self.step_ctr = torch.zeros(B, dtype=torch.int32, device=self.device)
        self.out_tokens = torch.full((B, max_steps), -1, dtype=torch.int32, device=self.device)
        self.logits = torch.empty((B, s.vocab), dtype=torch.float32, device=self.device)
        cap = model.max_pages * model.page_size
        self.rope = rope_table(cap, s.head_dim, s.rope_theta, self.device)
        n_pages = int(model.k_cache[0].shape[0])
        a = StepArgs()
        a.layers = C.cast(self._layer_arr, _vp)
        a.n_layers = L
        a.embed = _p(model.embed)
        a.final_norm = _p(model.final_norm)
        a.lm_head = _p(model.lm_head)
        a.lm_head_scales = _p(model.lm_head_scales)
        a.lm_act = act if lm_act is None else lm_act
        a.vocab = s.vocab
        a.k_cache = C.cast(self._k_arr, _vp)
        a.v_cache = C.cast(self._v_arr, _vp)
        a.page_table = _p(model.page_table)
        a.page_size = model.page_size
        a.max_pages = model.max_pages
        a.n_pages = n_pages
        a.rope_table = _p(self.rope)
        a.rope_max_pos = cap
        a.tok, a.pos, a.step, a.out_tokens = _p(self.tok), _p(self.pos), _p(self.step_ctr), _p(self.out_tokens)
        a.max_steps = max_steps
        a.batch = B
        a.logits = _p(self.logits)
        a.lm_wtype = QD_W_INT4 if model.lm_head.dtype == torch.uint8 else QD_W_BF16
        a.top_k = top_k
        if top_k:
            self.topk_ids = torch.full((top_k,), -1, dtype=torch.int32, device=self.device)
            self.topk_vals = torch.zeros(top_k, dtype=torch.float32, device=self.device)
            a.topk_ids, a.topk_vals = _p(self.topk_ids), _p(self.topk_vals)
        self.args = a
        nbytes = int(lib().qd_step_workspace_bytes(C.byref(a)))
        if verify_k:  # room for speculative verify passes of up to verify_k tokens
            nbytes = max(nbytes, int(lib().qd_verify_workspace_bytes(C.byref(a), verify_k)))
            self.verify_logits = torch.empty((verify_k, s.vocab), dtype=torch.float32, device=self.device)
            self.verify_target = torch.zeros(verify_k, dtype=torch.int32, device=self.device)
            self.n_accept = torch.zeros(1, dtype=torch.int32, device=self.device)
        if prefill_max:  # room for prompts of up to prefill_max tokens
            nbytes = max(nbytes, int(lib().qd_prefill_workspace_bytes(C.byref(a), prefill_max)))
            self.prefill_logits = torch.empty(s.vocab, dtype=torch.float32, device=self.device)
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=self.device)
        a.workspace = _p(self.workspace)
        a.workspace_bytes = nbytes
        self._graph = None

    @property
    def launches_per_step(self) -> int:
        return int(lib().qd_step_launch_count(C.byref(self.args)))

    def residual(self) -> torch.Tensor:
        """The f32 residual stream [B, H] left in the workspace by the last step."""
        H = self.m.shape.hidden
        return self.workspace[: self.batch * H * 4].view(torch.float32).view(self.batch, H)

    def rows_residual(self, n: int) -> torch.Tensor:
        """The f32 residual rows [n, H] of the last verify pass or prefill (their scratch
        follows the decode step's workspace)."""
        H = self.m.shape.hidden
        off = int(lib().qd_step_workspace_bytes(C.byref(self.args)))
        return self.workspace[off: off + n * H * 4].view(torch.float32).view(n, H)

    def step(self, stream=None):
        _check(lib().qd_decode_step(C.byref(self.args), _stream(stream)))

    def verify(self, draft, stream=None):
        """One speculative verify pass over tok and the k - 1 draft tokens (device int32):
        fills verify_logits[:k], verify_target[:k] and n_accept, and advances the state."""
        k = int(draft.numel()) + 1
        _check(lib().qd_verify_step(C.byref(self.args), _p(draft) if k > 1 else None, k, _p(self.verify_logits),
                                    _p(self.verify_target), _p(self.n_accept), _stream(stream)))

    def prefill(self, tokens, stream=None):
        """The prompt `tokens` (device int32 [n]) at positions pos .. pos + n - 1 in one
        pass: writes their K/V, fills prefill_logits with the last row's logits and
        advances the state (tok = its argmax, pos += n, step += 1)."""
        _check(lib().qd_prefill(C.byref(self.args), _p(tokens), int(tokens.numel()), _p(self.prefill_logits),
                                _stream(stream)))

    def capture(self, steps_per_launch: int, stream=None):
        if self._graph is not None:
            lib().qd_graph_destroy(self._graph)
        g = _vp()
        _check(lib().qd_graph_create(C.byref(self.args), steps_per_launch, _stream(stream), C.byref(g)))
        self._graph = g
        self.graph_steps = steps_per_launch

    def replay(self, stream=None):
        _check(lib().qd_graph_launch(self._graph, _stream(stream)))

    def close(self):
        if self._graph is not None:
            lib().qd_graph_destroy(self._graph)
            self._graph = None
        for h in self._handles:
            lib().qd_destroy_layer(h)
        self._handles = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
