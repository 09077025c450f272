"""CPU checks of the C-ABI library: it builds for sm_103a, loads, exports every
function include/qd.h declares, the ctypes structs match the C layout, and the
host-side argument validation rejects bad calls before touching the GPU."""
import ctypes as C
import os
import subprocess

import pytest

from transformer_decode_step_weight_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api.lib()


def test_every_header_function_is_exported_and_bound(lib):
    names = api.header_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
        assert n in api._SIGS, f"{n} has no ctypes signature"


def test_struct_layout_matches_c(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "qd.h"
int main(void) {
  printf("%zu %zu %zu\n", sizeof(qd_layer_dims), sizeof(qd_layer_weights), sizeof(qd_step_args));
  printf("%zu %zu %zu %zu %zu\n", offsetof(qd_step_args, rope_table), offsetof(qd_step_args, tok),
         offsetof(qd_step_args, max_steps), offsetof(qd_step_args, logits), offsetof(qd_step_args, workspace_bytes));
  return 0;
}
''')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-I", "/usr/local/cuda/include", str(src), "-o",
                    str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    sizes = [int(v) for v in out[:3]]
    offs = [int(v) for v in out[3:]]
    assert sizes == [C.sizeof(api.LayerDims), C.sizeof(api.LayerWeights), C.sizeof(api.StepArgs)]
    S = api.StepArgs
    assert offs == [S.rope_table.offset, S.tok.offset, S.max_steps.offset, S.logits.offset,
                    S.workspace_bytes.offset]


def test_host_validation_without_gpu(lib):
    # null pointers and bad sizes are rejected on the host, before any CUDA call
    assert lib.qd_gemv_bf16(None, 10, 16, None, 0, None, 1, None) == -1
    assert b"null" in lib.qd_last_error()
    assert lib.qd_gemv_q8_0(None, None, 4, 33, None, None, None, 0, None, None) == -1
    assert lib.qd_quantize_q8_0(None, 32, None, None, None) == -1
    d = api.LayerDims(1024, 16, 8, 64, 3072, 1e-6, 1e6, 0, 0)
    w = api.LayerWeights()
    h = C.c_void_p()
    assert lib.qd_create_layer(C.byref(d), C.byref(w), C.byref(h)) == -2      # head_dim 64 unsupported
    d.head_dim = 128
    assert lib.qd_create_layer(C.byref(d), C.byref(w), C.byref(h)) == -1      # null weights
    d.n_q_heads = 12
    assert lib.qd_create_layer(C.byref(d), C.byref(w), C.byref(h)) == -1      # Hq % Hkv != 0
    assert lib.qd_decode_step(None, None) == -1
    assert lib.qd_prefill(None, None, 4, None, None) == -1
    assert lib.qd_prefill_workspace_bytes(None, 4) == 0
    assert lib.qd_debug_wait_timeout(0, None) == -1      # the limit is checked on the host
    # the batched Q8_0 GEMM: null pointers, cols not a multiple of 32, and cols that are a
    # multiple of 32 but not of 256 (its scale boxes) are refused before any launch;
    # the non-null pointers below are never dereferenced
    fake = C.c_void_p(1 << 20)
    assert lib.qd_gemm_q8_0(None, None, 128, 256, None, 2, None, None, 0, None) == -1
    assert lib.qd_gemm_q8_0(fake, fake, 128, 300, fake, 2, fake, None, 0, None) == -1
    assert lib.qd_gemm_q8_0(fake, fake, 128, 288, fake, 2, fake, None, 0, None) == -2
    assert b"256" in lib.qd_last_error()
    assert lib.qd_gemm_q8_0(fake, fake, 128, 256, fake, 0, fake, None, 0, None) == -1    # batch 0
    # workspace sizing is pure host arithmetic
    assert lib.qd_attn_workspace_bytes(1, 32, 8, 4224) > 0
    assert lib.qd_attn_workspace_bytes(0, 32, 8, 4224) == 0
    assert lib.qd_argmax_workspace_bytes(64) > lib.qd_argmax_workspace_bytes(1)


def test_api_refuses_to_run_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(api, "_lib", None)
    monkeypatch.setattr(api, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        api.lib()
