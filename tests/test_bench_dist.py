"""The multi-process side of bench.py on CPU (gloo, world size 2): rank setup from
the torchrun environment, the barrier, max-over-ranks timing, and the reference
arm's rule that only rank 0 works."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist, r, w, local = bench.dist_setup(None)
    assert dist is not None and r == rank and w == world and local == rank
    bench.barrier(dist)
    got = bench.max_over_ranks(dist, 1.5 + rank)          # each rank's elapsed time
    dist.destroy_process_group()
    q.put((rank, got))


def test_two_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert res == [(0, 2.5), (1, 2.5)]


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], capture_output=True, text=True, env=env, timeout=300)
    assert out.returncode == 0
    assert out.stdout.strip() == ""


def test_weight_byte_accounting_matches_the_shapes():
    sys.path.insert(0, ROOT)
    import bench
    from transformer_decode_step_weight_gb300 import synth
    s = synth.QWEN3_8B
    wb = bench.weight_bytes(s, "bf16")
    # 36 x (6144 + 4096 + 24576) x 4096 + 4096 x 12288, 2 bytes each, + LM head 151936 x 4096 x 2
    layers = 36 * ((6144 + 4096 + 24576) * 4096 + 4096 * 12288) * 2
    assert wb - layers - 151936 * 4096 * 2 == 36 * (2 * 4096 + 2 * 128) * 2 + 2 * 4096 * 2
    assert bench.kv_bytes(s, 4095) == 36 * 8 * 128 * 2 * 2 * 4096
    q8 = bench.weight_bytes(s, "q8_0")
    assert abs(q8 / wb - 1.0625 / 2) < 1e-3
    # INT4: half a byte per weight plus one 2-byte scale per output row
    w4 = bench.weight_bytes(s, "int4")
    rows = 36 * (6144 + 4096 + 24576 + 4096) + 151936
    assert w4 - layers // 4 - 151936 * 4096 // 2 - rows * 2 == 36 * (2 * 4096 + 2 * 128) * 2 + 2 * 4096 * 2


@pytest.mark.parametrize("name", ["qwen3-8b-bf16", "qwen3-0.6b", "qwen3-8b-q8_0", "qwen3-8b-int4",
                                  "qwen3-8b-bf16-paged-b64", "qwen3-8b-q8_0-paged-b64"])
def test_workloads_are_the_named_shapes(name):
    from transformer_decode_step_weight_gb300 import synth
    wl = synth.WORKLOADS[name]
    assert wl.shape.head_dim == 128 and wl.shape.vocab == 151936
    assert wl.shape.n_q_heads % wl.shape.n_kv_heads == 0


@pytest.mark.parametrize("deq,act,want", [(None, "f32", ("f32", "f32")), (None, "i8", ("i8", "i8")),
                                          (0, "f32", ("i8", "i8")), (1, "f32", ("i8", "f32")),
                                          (2, "i8", ("f32", "f32"))])
def test_q8_deq_levels_pick_the_lanes(deq, act, want):
    # deq 0: dp4a everywhere; 1: dp4a in the layers, f32 activations for the LM head;
    # 2: f32 activations everywhere; without --deq, --act sets both
    import types
    sys.path.insert(0, ROOT)
    import bench
    assert bench.q8_lanes(types.SimpleNamespace(deq=deq, act=act)) == want


def test_dtype_labels_name_the_arithmetic():
    sys.path.insert(0, ROOT)
    import bench
    from transformer_decode_step_weight_gb300 import synth
    wl = synth.WORKLOADS
    assert bench.dtype_label(wl["qwen3-8b-bf16"], "f32", "f32") == "bf16"
    assert bench.dtype_label(wl["qwen3-8b-q8_0"], "i8", "i8") == "q8_0/i8"
    assert bench.dtype_label(wl["qwen3-8b-q8_0"], "i8", "f32") == "q8_0/i8+head_f32"
    assert bench.dtype_label(wl["qwen3-8b-q8_0-paged-b64"], "f32", "f32") == "q8_0->bf16"
    assert bench.q8_lane_label(wl["qwen3-8b-bf16-paged-b64"], "f32", "f32") is None
