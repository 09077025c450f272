"""Decode-step benchmark: Qwen3-8B-shaped BF16 greedy decode at batch 1.

One step = one token through the whole path: embedding gather, every decoder
layer (RMSNorm + QKV GEMV, QK-norm + RoPE + K/V write + split-KV attention,
O GEMV + residual, RMSNorm + gate/up GEMV, SwiGLU + down GEMV + residual), the
final RMSNorm + LM-head GEMV and the on-device argmax that advances token and
position, replayed as one captured CUDA graph per step. The workload runs 128
greedy steps from context 4096; longer timed runs restart it every 128 steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). Multi-GPU runs (torchrun) are independent
replicas, one sequence per GPU, no collective on the data path.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from transformer_decode_step_weight_gb300 import synth  # noqa: E402

METRIC = "Qwen3-8B-shape decode tok/s @bs1; achieved HBM GB/s vs GB300 peak"
BAD_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--reps", type=int, default=5, help="timed repetitions of K steps; value is their median")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3-8b-bf16",
                    choices=["qwen3-8b-bf16", "qwen3-0.6b", "qwen3-8b-q8_0", "qwen3-8b-int4",
                             "qwen3-8b-bf16-b2", "qwen3-8b-bf16-b4", "qwen3-8b-bf16-b8",
                             "qwen3-8b-bf16-paged-b64", "qwen3-8b-q8_0-paged-b64", "qwen3-0.6b-layer"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=128)
    ap.add_argument("--no-probe", action="store_true", help="skip the dominant-kernel event probe")
    ap.add_argument("--kernel", choices=["gemv_bf16", "gemv_q8_f32", "gemv_q8_i8", "gemv_w4", "gemv_w4_topk",
                                         "attention", "attention_batched", "gemm_tc", "gemm_q8"],
                    help="time one kernel alone on a full-size shape (profiling aid) instead of the step")
    ap.add_argument("--rows", type=int, default=24576)
    ap.add_argument("--cols", type=int, default=4096)
    ap.add_argument("--ctx", type=int, default=4224)
    ap.add_argument("--batch", type=int, default=64,
                    help="rows of x for --kernel gemm_tc; sequences for --kernel attention_batched")
    ap.add_argument("--act", choices=["f32", "i8"], default="f32", help="Q8_0 activation lane (batch 1)")
    ap.add_argument("--prefill", type=int, default=0, metavar="N",
                    help="time the prefill of an N-token prompt (positions 0 .. N-1) instead of decode")
    ap.add_argument("--verify", type=int, default=0, metavar="K",
                    help="time speculative verify passes of K tokens (K - 1 drafts) against K single-token steps "
                         "on the batch-1 workload")
    ap.add_argument("--layers", type=int, default=0, metavar="N",
                    help="--verify and --prefill: a model of N decoder layers instead of the workload's "
                         "(profiling aid)")
    ap.add_argument("--deq", type=int, choices=[0, 1, 2],
                    help="Q8_0 lanes by level: 0 = dp4a everywhere, 1 = dp4a in the layers and f32 activations for "
                         "the LM head, 2 = f32 activations everywhere (overrides --act)")
    return ap.parse_args()


def q8_lanes(args):
    """(layer lane, LM-head lane) names of the Q8_0 batch-1 GEMVs."""
    if args.deq is not None:
        return ("i8", "i8") if args.deq == 0 else (("i8", "f32") if args.deq == 1 else ("f32", "f32"))
    return args.act, args.act


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return dist, rank, world, local
    return None, rank, world, local


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.rows = []
        self.proc = None
        self.idx = device_index

    def start(self):
        try:
            bus = torch.cuda.get_device_properties(self.idx).pci_bus_id
            sel = ["-i", bus] if bus else []
        except Exception:
            sel = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", *sel, f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.th.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- byte accounting


def weight_bytes(s: synth.Shape, wtype: str) -> int:
    """Bytes of weights one token streams: every projection, the LM head, norms, one embedding row.
    BF16: 2 B per weight; Q8_0: 34 B per 32 weights; INT4: 0.5 B per weight plus a 2-byte
    scale per output row."""
    mats = [(s.qkv_rows, s.hidden), (s.hidden, s.n_q_heads * s.head_dim), (2 * s.ffn, s.hidden),
            (s.hidden, s.ffn)]

    def mbytes(r, k):
        if wtype == "bf16":
            return r * k * 2.0
        if wtype == "q8_0":
            return r * k * 34.0 / 32.0
        return r * k * 0.5 + r * 2.0

    layer = sum(mbytes(r, k) for r, k in mats) + (2 * s.hidden + 2 * s.head_dim) * 2
    return int(s.n_layers * layer + mbytes(s.vocab, s.hidden) + s.hidden * 2 + s.hidden * 2)


def kv_bytes(s: synth.Shape, pos: int) -> int:
    """K/V bytes one step at position `pos` reads (pos tokens) and writes (1 token), all layers."""
    row = s.n_kv_heads * s.head_dim * 2 * 2       # K and V, bf16
    return s.n_layers * row * (pos + 1)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def tensor_peak(sustained: bool):
    """The measured dense bf16 tensor peak in TFLOP/s (burst, or the seconds-long
    sustained figure for kernels timed inside a long run)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops_sustained" if sustained else "bf16_tflops"]), "measured"
    except Exception:
        return (1700.0 if sustained else 1900.0), "fallback"


def traffic_record(kernel_src: str):
    """DRAM traffic per launch of the dominant kernel from the committed ncu summary,
    valid only while the kernel source is unchanged since the counters were taken."""
    stem = os.path.splitext(os.path.basename(kernel_src))[0]
    path = os.path.join(ROOT, "profiles", f"{stem}_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        with open(kernel_src, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()[:16]
        if rec.get("source_sha") != sha:
            return None
        return rec
    except Exception:
        return None


# ---------------------------------------------------------------- oracle inputs
# Host copies of the seeded tensors in the oracle's form (bit views, no arithmetic),
# for the CPU-baseline leg and the reference arm, the only places the bench runs the
# oracle.


def _oracle_dims(oracle, s: synth.Shape):
    return oracle.Dims(s.hidden, s.n_q_heads, s.n_kv_heads, s.head_dim, s.ffn, s.rms_eps, s.rope_theta)


def _oracle_layer(oracle, lt: synth.LayerTensors, wtype: str):
    mats = ("w_qkv", "w_o", "w_gu", "w_down")
    if wtype == "bf16":
        w, sc = {k: synth.bits_u16(getattr(lt, k)) for k in mats}, {}
    else:
        host = synth.host_u8 if wtype == "int4" else synth.host_i8
        w = {k: host(getattr(lt, k)) for k in mats}
        sc = {k: synth.bits_u16(getattr(lt, k)) for k in ("s_qkv", "s_o", "s_gu", "s_down")}
    n = {k: synth.bits_u16(getattr(lt, k)) for k in ("ln_in", "ln_post", "q_norm", "k_norm")}
    return oracle.LayerWeights(**w, **n, **sc)


def _oracle_lane(mt, wl, q8_act: str = "f32"):
    """(mode, act) of the oracle lane that the GPU step runs for this workload."""
    if mt.wtype == "bf16":
        mode, act = "bf16", "bf16"
    elif mt.wtype == "int4":
        mode, act = "bf16", "w4"
    else:  # the Q8_0 lane the GPU step runs at the workload's batch
        mode, act = ("bf16", "w_bf16") if wl.batch > 1 else ("f32", q8_act)
    return mode, act


def _oracle_lm_rows(mt, idx):
    """The LM head's rows `idx` (and their scales) as the oracle takes them."""
    if mt.lm_head_scales is None:
        return synth.bits_u16(mt.lm_head[idx]), None
    host = synth.host_u8 if mt.lm_head.dtype == torch.uint8 else synth.host_i8
    return host(mt.lm_head[idx]), synth.bits_u16(mt.lm_head_scales[idx])


def _oracle_cache0(oracle, mt, n_tokens: int):
    """Layer 0's logical float64 [Hkv, n_tokens, D] K and V of sequence 0 (slots past the
    cached length zero)."""
    pt = mt.page_table[0].cpu().numpy()
    have = int(mt.seq_lens[0])
    out = []
    for c in (mt.k_cache[0], mt.v_cache[0]):
        x = oracle.bf16_to_f64(oracle.gather_paged(synth.bits_u16(c), pt, have))
        full = np.zeros((x.shape[0], n_tokens, x.shape[2]))
        full[:, :have] = x
        out.append(full)
    return out


# ---------------------------------------------------------------- our arm


def run_ours(args, dist, rank, world, local):
    from transformer_decode_step_weight_gb300 import api
    from transformer_decode_step_weight_gb300 import build as b

    b.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = synth.WORKLOADS[args.workload]
    s = wl.shape
    run_len = wl.steps
    mt = synth.make_model(s, wl.wtype, args.seed + rank, dev, batch=wl.batch, ctx=None if wl.paged else wl.ctx,
                          steps=run_len, paged=wl.paged)
    act, lm_act = q8_lanes(args)
    lane = api.QD_ACT_I8 if act == "i8" else api.QD_ACT_F32
    lm_lane = api.QD_ACT_I8 if lm_act == "i8" else api.QD_ACT_F32
    dec = api.Decoder(mt, max_steps=run_len, act=lane, lm_act=lm_lane, device=dev)
    lens = [int(v) for v in mt.seq_lens.cpu()]
    tok0, pos0 = dec.tok.clone(), dec.pos.clone()

    def reset():
        dec.tok.copy_(tok0)
        dec.pos.copy_(pos0)
        dec.step_ctr.zero_()

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        dec.capture(1)
        for _ in range(args.warmup):
            dec.replay()
        reset()
    stream.synchronize()
    assert api.check_device_error(stream) == 0

    # ---- timed region: `reps` repetitions of K graph replays (one token each); the
    # decode run continues across repetitions (restarting every run_len steps), so the
    # repetitions cover successive positions. Each has its own clock samples.
    K = args.steps
    reps = max(1, args.reps)
    rep_ms, rep_clk, rep_bytes = [], [], []
    wb = weight_bytes(s, wl.wtype)
    done = 0
    for _ in range(reps):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clocks = ClockSampler(local)
        barrier(dist)
        torch.cuda.synchronize(dev)
        clocks.start()
        time.sleep(0.3)
        idx = []
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(K):
                if done and done % run_len == 0:
                    reset()
                idx.append(done % run_len)
                dec.replay()
                done += 1
            ev1.record(stream)
        stream.synchronize()
        torch.cuda.synchronize(dev)
        rep_clk.append(clocks.stop())
        barrier(dist)
        rep_ms.append(max_over_ranks(dist, ev0.elapsed_time(ev1)))
        rep_bytes.append(sum(wb + sum(kv_bytes(s, n + i) for n in lens) for i in idx))
    assert api.check_device_error(stream) == 0
    order = sorted(range(reps), key=lambda r: rep_ms[r])
    med = order[reps // 2]
    ms_max = rep_ms[med]
    ms = ms_max
    clk = dict(rep_clk[med])
    clk["per_repetition"] = [{"sm_mhz": c["sm_mhz"], "reasons": c["reasons"]} for c in rep_clk]
    clk["reasons"] = sorted({r for c in rep_clk for r in c["reasons"]})
    toks = K * dec.batch * world
    value = toks / (ms_max / 1e3)
    rep_tok_s = [toks / (m / 1e3) for m in rep_ms]
    # algorithmic bytes of the timed steps (the median repetition's positions)
    hbm_peak, peak_kind = peaks()
    step_gbs = rep_bytes[med] / (ms / 1e3) / 1e9

    # ---- a pure-read streaming peak on this GPU (a 4 GiB reduction), for the third
    # denominator of the step's fraction (the others: the measured copy peak, 8 TB/s)
    read_peak = measure_read_peak(dev, stream)

    # ---- dominant kernel: the BF16 GEMV, every launch of one token, events on its stream
    roof = None
    if not args.no_probe and ((wl.batch == 1 and wl.wtype in ("bf16", "int4")) or
                              (wl.wtype == "bf16" and 2 <= wl.batch <= 8)):
        roof = dominant_kernel_roofline(api, mt, s, stream, hbm_peak, peak_kind, batch=wl.batch)

    # ---- end to end through the public API: per step H2D of the input token/position
    # from pinned memory, the step, D2H of the next token, host reads it
    e2e = run_e2e(dec, stream, args.e2e_steps, reset, dist, world, run_len)
    launches = K * dec.launches_per_step   # in one timed repetition

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(mt, s, wl, lens[0])

    if rank == 0:
        out = {
            "metric": METRIC, "value": round(value, 3), "unit": "tok/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(ms_max / K, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dtype_label(wl, act, lm_act),
            "data": "synthetic",
            "config": {"workload": wl.name, "description": wl.description, "global_batch": dec.batch * world,
                       "q8_lane": q8_lane_label(wl, act, lm_act),
                       "ctx_start": wl.ctx if not wl.paged else "uniform[128,4096]", "decode_run_steps": run_len,
                       "parallelism": f"replicas x{world}",
                       "graph": "one CUDA graph per step, PDL between kernels",
                       "l2": f"inputs larger than L2 ({wb / 1e9:.1f} GB of weights streamed per step)"},
            "roofline": roof,
            "step_roofline": {"bound": "hbm", "achieved": round(step_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                              "frac": round(step_gbs / hbm_peak, 4), "peak_kind": peak_kind,
                              "frac_of_nominal_8tbs": round(step_gbs / 8000.0, 4),
                              "read_peak_gbs": read_peak,
                              "frac_of_read_peak": round(step_gbs / read_peak, 4) if read_peak else None,
                              "bytes_per_step": int(rep_bytes[med] / K)},
            "repetitions": {"n": reps, "steps_each": K, "tok_s": [round(v, 3) for v in rep_tok_s],
                            "median": round(value, 3), "min": round(min(rep_tok_s), 3),
                            "max": round(max(rep_tok_s), 3)},
            "e2e": e2e, "gpu_launches": launches, "clocks": clk, "cpu_baseline": cpu,
        }
        print(json.dumps(out), flush=True)
    dec.close()


def dtype_label(wl, act, lm_act):
    """The arithmetic the step computes in: bf16 MMA / FMA, or the Q8_0 lanes."""
    if wl.wtype == "bf16":
        return "bf16"
    if wl.wtype == "int4":
        return "int4 weights x bf16 activations (f32 accumulate)"
    if wl.batch > 1:
        return "q8_0->bf16"          # weights widened on chip, bf16 tensor-core MMA
    return f"q8_0/{act}" if act == lm_act else f"q8_0/{act}+head_{lm_act}"


def q8_lane_label(wl, act, lm_act):
    if wl.wtype != "q8_0":
        return None
    if wl.batch > 1:
        return "weights widened to bf16 on chip (tensor cores)"
    return act if act == lm_act else f"{act} (LM head {lm_act})"


def measure_read_peak(dev, stream, gib=4, reps=5):
    """Pure-read HBM bandwidth: best of `reps` sums over a `gib` GiB f32 buffer (read once
    per sum, far larger than L2), timed with CUDA events on `stream`. None if it cannot run."""
    try:
        buf = torch.ones(gib * (1 << 28), dtype=torch.float32, device=dev)
        best = None
        with torch.cuda.stream(stream):
            buf.sum()
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                buf.sum()
                e1.record(stream)
                e1.synchronize()
                ms = e0.elapsed_time(e1)
                best = ms if best is None or ms < best else best
        del buf
        return round(gib * (1 << 30) / (best / 1e3) / 1e9, 1)
    except Exception:
        return None


def dominant_kernel_roofline(api, mt, s, stream, hbm_peak, peak_kind, batch=1):
    """Average duration of the weight GEMV's launches over one step's projections, timed
    with CUDA events on the stream they run on, three passes; algorithmic bytes = the
    weight bytes (and, for INT4, the per-row scales) each launch reads. Batch 1: the
    ring GEMV's K = hidden launches (36 x QKV, O, gate+up, and the LM head); batch 2..8:
    the mma.sync GEMV over `batch` activation rows, every projection (down included)."""
    B = batch
    x = torch.randn((B, max(s.hidden, s.n_q_heads * s.head_dim, s.ffn)),
                    device=mt.embed.device).to(torch.bfloat16)
    xo = x[:, : s.n_q_heads * s.head_dim].contiguous()
    xh = x[:, : s.hidden].contiguous()
    xf = x[:, : s.ffn].contiguous()
    w4 = mt.wtype == "int4"
    mats = []
    for lt in mt.layers:
        if w4:
            mats += [(lt.w_qkv, lt.s_qkv, xh[0]), (lt.w_o, lt.s_o, xo[0]), (lt.w_gu, lt.s_gu, xh[0])]
        else:
            mats += [(lt.w_qkv, None, xh), (lt.w_o, None, xo), (lt.w_gu, None, xh)]
            if B > 1:
                mats.append((lt.w_down, None, xf))
    mats.append((mt.lm_head, mt.lm_head_scales, xh[0] if w4 else xh))
    ys = {id(w): torch.empty((B, w.shape[0]), dtype=torch.float32, device=x.device) for w, _, _ in mats}

    w4ws = {}
    if w4:   # the step's split-K workspace, one per shape
        for w, _, _ in mats:
            nb = api.gemv_w4_workspace_bytes(w.shape[0], 2 * w.shape[1])
            w4ws[tuple(w.shape)] = torch.zeros(max(nb, 16), dtype=torch.uint8, device=x.device) if nb else None

    def run(w, sc, xx):
        if w4:
            api.gemv_w4(w, sc, xx, ys[id(w)][0], workspace=w4ws[tuple(w.shape)], stream=stream)
        else:
            api.gemv_bf16(w, xx, ys[id(w)], stream=stream)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for m in mats:   # warm
            run(*m)
        e0.record(stream)
        for _ in range(3):
            for m in mats:
                run(*m)
        e1.record(stream)
    stream.synchronize()
    ms = e0.elapsed_time(e1)
    n = 3 * len(mats)
    if w4:
        bytes_per_launch = sum(w.numel() + 2 * w.shape[0] for w, _, _ in mats) / len(mats)
    else:
        bytes_per_launch = sum(w.numel() * 2 for w, _, _ in mats) / len(mats)
    avg_s = ms / 1e3 / n
    achieved = bytes_per_launch / avg_s / 1e9
    src = "gemv_w4.cu" if w4 else "gemv_bf16.cu" if B == 1 else "gemv_mma.cu"
    rec = traffic_record(os.path.join(ROOT, "transformer_decode_step_weight_gb300", "csrc", src))
    traffic = None
    if rec is not None:
        traffic = rec.get("traffic_bytes_per_launch")
    if B > 1:
        kname, which = "gemv_mma_kernel", f"every projection of one step, {B} rows"
    else:
        kname, which = ("gemv_w4_kernel" if w4 else "gemv_bf16_kernel"), "K = hidden launches of one token"
    return {"bound": "hbm", "kernel": f"{kname} ({which})",
            "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
            "peak_kind": peak_kind, "avg_launch_us": round(avg_s * 1e6, 3),
            "algorithmic_bytes_per_launch": int(bytes_per_launch), "traffic": traffic}


def run_e2e(dec, stream, steps, reset, dist, world, run_len):
    """Host-driven loop through the public API: each step copies the input tokens and
    positions from pinned host memory, replays the step, copies the next tokens back
    and the host reads them before the next step."""
    if steps <= 0:
        return None
    B = dec.batch
    h_in = torch.empty((2, B), dtype=torch.int32, pin_memory=True)
    h_out = torch.empty(B, dtype=torch.int32, pin_memory=True)
    with torch.cuda.stream(stream):
        reset()
    stream.synchronize()
    h_in[0].copy_(dec.tok.cpu())
    h_in[1].copy_(dec.pos.cpu())
    barrier(dist)
    t0 = time.perf_counter()
    for i in range(steps):
        with torch.cuda.stream(stream):
            if i and i % run_len == 0:
                reset()
                stream.synchronize()
                h_in[0].copy_(dec.tok.cpu())
                h_in[1].copy_(dec.pos.cpu())
            dec.tok.copy_(h_in[0], non_blocking=True)
            dec.pos.copy_(h_in[1], non_blocking=True)
            dec.replay()
            h_out.copy_(dec.tok, non_blocking=True)
        stream.synchronize()
        h_in[0].copy_(h_out)
        h_in[1] += 1
    dt = time.perf_counter() - t0
    dt = max_over_ranks(dist, dt)
    return {"value": round(steps * B * world / dt, 3), "unit": "tok/s", "h2d_bytes_per_step": 8 * B,
            "d2h_bytes_per_step": 4 * B, "steps": steps}


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(mt, s, wl, ctx, n_layers_sample: int = 8):
    """The CPU oracle, as it stands, on a bounded sample: n full-size decoder layers
    (layer 0 of the model, at the workload's context) plus n/36 of the LM-head rows,
    scaled to one token."""
    import oracle
    torch.set_num_threads(_cores())
    od = _oracle_dims(oracle, s)
    ol = _oracle_layer(oracle, mt.layers[0], mt.wtype)
    k0, v0 = _oracle_cache0(oracle, mt, ctx + 1)
    x0 = oracle.bf16_to_f64(synth.bits_u16(mt.embed[int(mt.start_tok[0])]))
    frac = n_layers_sample / s.n_layers
    rows = np.arange(0, s.vocab, int(round(1 / frac)))
    idx = torch.as_tensor(rows, device=mt.lm_head.device)
    lm, lms = _oracle_lm_rows(mt, idx)
    mode, act = _oracle_lane(mt, wl)
    fn = synth.bits_u16(mt.final_norm)
    t0 = time.perf_counter()
    res = x0
    for _ in range(n_layers_sample):
        res = oracle.layer_step(od, ol, x0, k0, v0, ctx, mode=mode, act=act)
    xf = oracle.rmsnorm(res, oracle.bf16_to_f64(fn), s.rms_eps, mode)
    if lms is None:
        oracle.gemv_bf16(lm, xf)
    else:
        oracle.project(lm, lms, xf, act)
    dt = time.perf_counter() - t0
    sec_per_tok = dt / frac
    return {"value": round(1.0 / sec_per_tok, 5), "unit": "tok/s", "cores": _cores(), "kind": "oracle",
            "sample": f"{n_layers_sample} of {s.n_layers} full-size decoder layers at context {ctx} "
                      f"plus {len(rows)} of {s.vocab} LM-head rows ({dt:.1f} s), scaled to one token"}


# ---------------------------------------------------------------- reference arm


def run_reference(args, dist, rank, world, local):
    """The CPU oracle as it stands, on the host cores: each step is one full-size
    decoder layer plus 1/36 of the LM-head rows (1/36 of one token's work)."""
    if rank != 0:
        return
    import oracle
    wl = synth.WORKLOADS[args.workload]
    s = wl.shape
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    mt = synth.make_model(s, wl.wtype, args.seed, dev, n_layers=1, ctx=wl.ctx, steps=1)
    torch.set_num_threads(_cores())
    od = _oracle_dims(oracle, s)
    ol = _oracle_layer(oracle, mt.layers[0], wl.wtype)
    k0, v0 = _oracle_cache0(oracle, mt, wl.ctx + 1)
    x0 = oracle.bf16_to_f64(synth.bits_u16(mt.embed[int(mt.start_tok[0])]))
    rows = np.arange(0, s.vocab, s.n_layers)
    idx = torch.as_tensor(rows, device=mt.lm_head.device)
    mode, act = _oracle_lane(mt, wl, q8_lanes(args)[0])
    lm, lms = _oracle_lm_rows(mt, idx)
    fn = oracle.bf16_to_f64(synth.bits_u16(mt.final_norm))
    del mt

    def one():
        r = oracle.layer_step(od, ol, x0, k0, v0, wl.ctx, mode=mode, act=act)
        xf = oracle.rmsnorm(r, fn, s.rms_eps, mode)
        if lms is None:
            oracle.gemv_bf16(lm, xf)
        else:
            oracle.project(lm, lms, xf, act)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt = time.perf_counter() - t0
    tok_s = args.steps / s.n_layers / dt
    sample = (f"each step: 1 of {s.n_layers} full-size decoder layers at context {wl.ctx} + {len(rows)} of "
              f"{s.vocab} LM-head rows (1/{s.n_layers} of a token)")
    out = {"impl": "reference", "metric": METRIC, "value": round(tok_s, 5), "unit": "tok/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": wl.name, "description": wl.description, "global_batch": 1},
           "cpu_baseline": {"value": round(tok_s, 5), "unit": "tok/s", "cores": _cores(), "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": round(tok_s, 5), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_kernel(args):
    """One kernel alone, `steps` launches on distinct buffers larger than L2 where the
    shape allows, timed with CUDA events; prints achieved GB/s of algorithmic bytes."""
    from transformer_decode_step_weight_gb300 import api
    from transformer_decode_step_weight_gb300 import build as b
    b.build()
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(args.seed)
    R, K = args.rows, args.cols
    stream = torch.cuda.Stream(device=dev)
    copies = max(1, min(4, int(2 * 129e6 // max(1, R * K)) + 1))
    if args.kernel == "gemv_bf16":
        # --batch 1..8: x rows of the CUDA-core GEMV (larger batches take the tensor cores)
        nb = args.batch if 1 <= args.batch <= 8 else 1
        Ws = [(torch.randn((R, K), generator=g, device=dev) * 0.02).to(torch.bfloat16) for _ in range(copies)]
        x = torch.randn((nb, K), generator=g, device=dev).to(torch.bfloat16)
        y = torch.empty((nb, R), device=dev)
        nbytes = R * K * 2
        fn = lambda i: api.gemv_bf16(Ws[i % copies], x, y, stream=stream)  # noqa: E731
    elif args.kernel in ("gemv_q8_f32", "gemv_q8_i8"):
        qs = [torch.randint(-127, 128, (R, K), generator=g, device=dev, dtype=torch.int16).to(torch.int8)
              for _ in range(copies)]
        ds = [(torch.randn((R, K // 32), generator=g, device=dev).abs() * 0.002).to(torch.float16)
              for _ in range(copies)]
        x = torch.randn(K, generator=g, device=dev)
        y = torch.empty(R, device=dev)
        lane = api.QD_ACT_I8 if args.kernel.endswith("i8") else api.QD_ACT_F32
        nbytes = R * K + R * (K // 32) * 2
        fn = lambda i: api.gemv_q8_0(qs[i % copies], ds[i % copies], x=x, act=lane, y=y, stream=stream)  # noqa: E731
    elif args.kernel in ("gemv_w4", "gemv_w4_topk"):
        Ws = [torch.randint(0, 256, (R, K // 2), generator=g, device=dev, dtype=torch.int16).to(torch.uint8)
              for _ in range(copies)]
        ds = [(torch.randn(R, generator=g, device=dev).abs() * 0.01).to(torch.float16) for _ in range(copies)]
        x = torch.randn(K, generator=g, device=dev).to(torch.bfloat16)
        y = torch.empty(R, device=dev)
        nbytes = R * K // 2 + R * 2
        if args.kernel == "gemv_w4":
            wsb = api.gemv_w4_workspace_bytes(R, K)
            w4ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=dev) if wsb else None
            fn = lambda i: api.gemv_w4(Ws[i % copies], ds[i % copies], x, y, workspace=w4ws, stream=stream)  # noqa
        else:
            ws = torch.zeros(int(api.lib().qd_w4_topk_workspace_bytes()), dtype=torch.uint8, device=dev)
            fn = lambda i: api.gemv_w4_topk(Ws[i % copies], ds[i % copies], x, 8, y, ws, stream=stream)  # noqa
    elif args.kernel == "gemm_tc":
        Ws = [(torch.randn((R, K), generator=g, device=dev) * 0.02).to(torch.bfloat16) for _ in range(copies)]
        x = torch.randn((args.batch, K), generator=g, device=dev).to(torch.bfloat16)
        y = torch.empty((args.batch, R), device=dev)
        nbytes = R * K * 2
        fn = lambda i: api.gemv_bf16(Ws[i % copies], x, y, stream=stream)  # noqa: E731
    elif args.kernel == "gemm_q8":
        qs = [torch.randint(-127, 128, (R, K), generator=g, device=dev, dtype=torch.int16).to(torch.int8)
              for _ in range(copies)]
        ds = [(torch.randn((R, K // 32), generator=g, device=dev).abs() * 0.002).to(torch.float16)
              for _ in range(copies)]
        x = torch.randn((args.batch, K), generator=g, device=dev).to(torch.bfloat16)
        y = torch.empty((args.batch, R), device=dev)
        nb = api.gemm_workspace_bytes(R, K)
        ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device=dev) if nb else None
        nbytes = R * K + R * (K // 32) * 2
        fn = lambda i: api.gemm_q8_0(qs[i % copies], ds[i % copies], x, y=y, workspace=ws, stream=stream)  # noqa
    elif args.kernel == "attention_batched":
        # the batched workload's cache: `batch` sequences of 128..ctx tokens in 16-token
        # pages through a seeded random page table
        s = synth.QWEN3_8B
        B, ps = args.batch, 16
        lens = torch.randint(128, args.ctx + 1, (B,), generator=g, device=dev, dtype=torch.int64).to(torch.int32)
        per = [-(-int(v) // ps) for v in lens.cpu()]
        n_phys = sum(per)
        perm = torch.randperm(n_phys, generator=g, device=dev).to(torch.int32)
        pt = torch.zeros((B, max(per)), dtype=torch.int32, device=dev)
        off = 0
        for bi, npg in enumerate(per):
            pt[bi, :npg] = perm[off:off + npg]
            off += npg
        kp = torch.randn((n_phys, s.n_kv_heads, ps, 128), generator=g, device=dev).to(torch.bfloat16)
        vp = torch.randn((n_phys, s.n_kv_heads, ps, 128), generator=g, device=dev).to(torch.bfloat16)
        q = torch.randn((B, s.n_q_heads, 128), generator=g, device=dev)
        out = torch.empty_like(q)
        ws = torch.zeros(api.attn_workspace_bytes(B, s.n_q_heads, s.n_kv_heads, max(per) * ps), dtype=torch.uint8,
                         device=dev)
        nbytes = int(lens.sum()) * s.n_kv_heads * 128 * 2 * 2
        fn = lambda i: api.attn_decode_paged(q, kp, vp, pt, lens, 0.0884, out=out, workspace=ws, stream=stream)  # noqa
    else:
        s = synth.QWEN3_8B
        n = args.ctx
        kp = torch.randn((1, s.n_kv_heads, n, 128), generator=g, device=dev).to(torch.bfloat16)
        vp = torch.randn((1, s.n_kv_heads, n, 128), generator=g, device=dev).to(torch.bfloat16)
        q = torch.randn((1, s.n_q_heads, 128), generator=g, device=dev)
        pt = torch.zeros((1, 1), dtype=torch.int32, device=dev)
        sl = torch.tensor([n], dtype=torch.int32, device=dev)
        out = torch.empty_like(q)
        ws = torch.zeros(api.attn_workspace_bytes(1, s.n_q_heads, s.n_kv_heads, n), dtype=torch.uint8, device=dev)
        nbytes = 2 * s.n_kv_heads * n * 128 * 2
        fn = lambda i: api.attn_decode_paged(q, kp, vp, pt, sl, 0.0884, out=out, workspace=ws, stream=stream)  # noqa
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            fn(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            fn(i)
        e1.record(stream)
    stream.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    peak, kind = peaks()
    gbs = nbytes / (ms / 1e3) / 1e9
    print(json.dumps({"kernel": args.kernel, "rows": R, "cols": K, "ctx": args.ctx, "us_per_launch": round(ms * 1e3, 3),
                      "algorithmic_bytes": nbytes, "achieved_gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                      "peak_kind": kind, "copies": copies}), flush=True)


def run_verify(args):
    """Speculative verify passes of k tokens (tok + k - 1 drafts, one sequence) against
    k plain decode steps, both as CUDA graphs on the batch-1 workload's model. Each
    verify replay restores the decode state first (three 4-byte copies), so every pass
    runs at the same positions; the drafts are random tokens (the pass costs the same
    whatever is accepted). Reports the pass latency and the tokens per second it would
    give if every draft were accepted."""
    from transformer_decode_step_weight_gb300 import api
    from transformer_decode_step_weight_gb300 import build as b
    b.build()
    dev = torch.device("cuda", 0)
    k = args.verify
    wl = synth.WORKLOADS[args.workload]
    assert wl.batch == 1, "speculative verify runs on one sequence"
    reps = max(1, args.reps)
    n = max(1, args.steps // 4)
    # room for every timed decode step (that leg does not restore the state)
    run_len = 4 * k + 16 + reps * (max(3, args.warmup) + n) + 8
    mt = synth.make_model(wl.shape, wl.wtype, args.seed, dev, ctx=wl.ctx, steps=run_len,
                          n_layers=args.layers if args.layers > 0 else None)
    act, lm_act = q8_lanes(args)
    dec = api.Decoder(mt, max_steps=run_len, act=api.QD_ACT_I8 if act == "i8" else api.QD_ACT_F32,
                      lm_act=api.QD_ACT_I8 if lm_act == "i8" else api.QD_ACT_F32, device=dev, verify_k=k)
    g = torch.Generator(device=dev)
    g.manual_seed(args.seed + 1)
    draft = torch.randint(0, wl.shape.vocab, (k - 1,), generator=g, device=dev, dtype=torch.int64).to(torch.int32)
    tok0, pos0 = dec.tok.clone(), dec.pos.clone()
    s = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s):
        dec.verify(draft, stream=s)
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        dec.tok.copy_(tok0)
        dec.pos.copy_(pos0)
        dec.step_ctr.zero_()
        dec.verify(draft, stream=s)

    def timed(fn, n):
        with torch.cuda.stream(s):
            for _ in range(max(3, args.warmup)):
                fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(n):
                fn()
            e1.record(s)
        s.synchronize()
        return e0.elapsed_time(e1) / n

    verify_ms = sorted(timed(graph.replay, n) for _ in range(reps))[reps // 2]
    with torch.cuda.stream(s):
        dec.tok.copy_(tok0)
        dec.pos.copy_(pos0)
        dec.step_ctr.zero_()
        dec.capture(1, stream=s)

    def one_step():
        dec.replay(stream=s)

    step_ms = sorted(timed(one_step, n) for _ in range(reps))[reps // 2]
    assert api.check_device_error(s) == 0
    out = {"metric": f"speculative verify pass, k = {k} tokens of one sequence", "value": round(k / (verify_ms / 1e3), 3),
           "unit": "tok/s if all k accepted", "ms_per_pass": round(verify_ms, 4),
           "ms_per_single_step": round(step_ms, 4), "pass_vs_k_steps": round(verify_ms / (k * step_ms), 4),
           "higher_is_better": True,
           "dtype": "bf16 mma.sync rows" if wl.wtype == "bf16" else "q8_0 widened to bf16, tcgen05 rows",
           "data": "synthetic", "config": {"workload": wl.name, "k": k, "drafts": "random tokens",
                                           "passes_timed": n, "repetitions": reps,
                                           "layers": args.layers or wl.shape.n_layers}}
    print(json.dumps(out), flush=True)
    dec.close()


def prefill_flops(s: synth.Shape, n: int, pos0: int = 0):
    """Algorithmic flops of one prefill: 2 per weight per row for the projections, the
    LM head for the last row, and the causal attention (q.k and p.v over the keys
    0 .. pos0 + i of row i, every q head)."""
    per_layer = (s.qkv_rows + 2 * s.ffn) * s.hidden + s.hidden * s.n_q_heads * s.head_dim + s.hidden * s.ffn
    gemm = 2.0 * n * per_layer * s.n_layers + 2.0 * s.vocab * s.hidden
    keys = n * pos0 + n * (n + 1) / 2
    attn = 4.0 * s.head_dim * s.n_q_heads * keys * s.n_layers
    return gemm, attn


def run_prefill_bench(args):
    """Prefill of one N-token prompt at positions 0 .. N - 1 on the workload's model,
    as a CUDA graph that restores the decode state first (three 4-byte copies), so every
    replay writes the same cache rows. Reports prompt tokens per second, the whole
    pass's achieved TFLOP/s, and the dominant kernel (the gate+up GEMM over the N rows)
    timed alone with CUDA events against the measured bf16 tensor peak."""
    from transformer_decode_step_weight_gb300 import api
    from transformer_decode_step_weight_gb300 import build as b
    b.build()
    dev = torch.device("cuda", 0)
    n = args.prefill
    wl = synth.WORKLOADS[args.workload]
    s = wl.shape
    assert wl.batch == 1 and wl.wtype in ("bf16", "q8_0"), "prefill runs on one sequence, BF16 or Q8_0 weights"
    mt = synth.make_model(s, wl.wtype, args.seed, dev, ctx=0, steps=n + 1,
                          n_layers=args.layers if args.layers > 0 else None)
    dec = api.Decoder(mt, max_steps=n + 1, device=dev, prefill_max=n)
    g = torch.Generator(device=dev)
    g.manual_seed(args.seed + 2)
    tokens = torch.randint(0, s.vocab, (n,), generator=g, device=dev, dtype=torch.int64).to(torch.int32)
    tok0, pos0 = dec.tok.clone(), dec.pos.clone()
    st = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(st):
        dec.prefill(tokens, stream=st)
    st.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        dec.tok.copy_(tok0)
        dec.pos.copy_(pos0)
        dec.step_ctr.zero_()
        dec.prefill(tokens, stream=st)

    def timed(fn, k):
        with torch.cuda.stream(st):
            for _ in range(max(3, args.warmup)):
                fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            for _ in range(k):
                fn()
            e1.record(st)
        st.synchronize()
        return e0.elapsed_time(e1) / k

    reps = max(1, args.reps)
    k = max(1, min(args.steps, 8))
    clocks = ClockSampler(0)
    clocks.start()
    ms_all = [timed(graph.replay, k) for _ in range(reps)]
    clk = clocks.stop()
    ms = sorted(ms_all)[reps // 2]
    assert api.check_device_error(st) == 0
    gemm_f, attn_f = prefill_flops(s, n)
    peak, kind = tensor_peak(sustained=True)
    total_tf = (gemm_f + attn_f) / (ms / 1e3) / 1e12
    # dominant kernel: the gate+up GEMM [2F, H] over the N rows, alone
    lt = mt.layers[0]
    x = torch.randn((n, s.hidden), generator=g, device=dev).to(torch.bfloat16)
    y = torch.empty((n, 2 * s.ffn), dtype=torch.float32, device=dev)
    widened = wl.wtype == "q8_0" and n > 128
    if wl.wtype == "bf16":
        fn = lambda: api.gemv_bf16(lt.w_gu, x, y, stream=st)  # noqa: E731
    elif widened:
        # above 128 rows the pass widens each projection's Q8_0 weights to bf16 and runs
        # the bf16 GEMM; the widened gate+up weights (built here with torch: an input only)
        wg = (lt.w_gu.float() * lt.s_gu.float().repeat_interleave(32, dim=1)).to(torch.bfloat16)
        fn = lambda: api.gemv_bf16(wg, x, y, stream=st)  # noqa: E731
    else:
        fn = lambda: api.gemm_q8_0(lt.w_gu, lt.s_gu, x, y, stream=st)  # noqa: E731
    gu_ms = sorted(timed(fn, 10) for _ in range(3))[1]
    gu_flops = 2.0 * n * 2 * s.ffn * s.hidden
    gu_tf = gu_flops / (gu_ms / 1e3) / 1e12
    bpeak, bkind = tensor_peak(sustained=False)
    out = {"metric": f"prefill of an {n}-token prompt (one sequence)", "value": round(n / (ms / 1e3), 1),
           "unit": "prompt tok/s", "ms_per_prefill": round(ms, 3), "higher_is_better": True,
           "dtype": ("bf16 tcgen05 GEMMs + bf16 mma.sync attention" if os.environ.get("QD_PREFILL_ATTN") == "mma" else "bf16 tcgen05 GEMMs + bf16 tcgen05 attention") if wl.wtype == "bf16" else
                    ("q8_0 widened to bf16 once per projection, tcgen05 GEMMs + bf16 tcgen05 attention" if widened else
                     "q8_0 widened to bf16 in the GEMM, tcgen05 GEMMs + bf16 tcgen05 attention"),
           "data": "synthetic",
           "config": {"workload": wl.name, "prompt_tokens": n, "positions": f"0..{n - 1}",
                      "graph": "one CUDA graph per prefill", "repetitions": reps, "prefills_each": k,
                      "layers": args.layers or s.n_layers},
           "roofline": {"bound": "tensor",
                        "kernel": (f"gemm_wide_kernel (the gate+up weights {2 * s.ffn} x {s.hidden} over {n} rows, f32 "
                                   "out; the pass runs these MMAs with the SwiGLU epilogue)") if wl.wtype == "bf16" else
                                  (f"gemm_wide_kernel (the gate+up weights widened from Q8_0, {2 * s.ffn} x {s.hidden} "
                                   f"over {n} rows)" if widened else
                                   f"gemm_tc_kernel Q8_0 (gate+up, {2 * s.ffn} x {s.hidden} x {n} rows)"),
                        "achieved": round(gu_tf, 1), "peak": bpeak, "unit": "TFLOP/s",
                        "frac": round(gu_tf / bpeak, 4), "peak_kind": f"{bkind} burst", "us_per_launch": round(gu_ms * 1e3, 2),
                        "traffic": None},
           "step_roofline": {"bound": "tensor", "achieved": round(total_tf, 1), "peak": peak, "unit": "TFLOP/s",
                             "frac": round(total_tf / peak, 4), "peak_kind": f"{kind} sustained",
                             "gemm_tflop": round(gemm_f / 1e12, 3), "attention_tflop": round(attn_f / 1e12, 3)},
           "repetitions": {"ms": [round(v, 3) for v in ms_all]},
           "clocks": clk}
    print(json.dumps(out), flush=True)
    dec.close()


def run_layer_bench(args):
    """One Qwen3-0.6B-shaped decoder layer at position 128 (the single-layer workload),
    timed with its weights coming from HBM: a 17-layer model (17 distinct random layers,
    535 MB, more than four times L2) and a 1-layer model of the same shape each replay
    their whole step as a CUDA graph, and the layer's time is the difference divided by
    16 (embedding, LM head and argmax cancel). Median of `reps` repetitions of each."""
    from transformer_decode_step_weight_gb300 import api
    from transformer_decode_step_weight_gb300 import build as b
    b.build()
    dev = torch.device("cuda", 0)
    wl = synth.WORKLOADS["qwen3-0.6b-layer"]
    s = wl.shape
    reps = max(1, args.reps)
    k = max(8, args.steps)
    run_len = reps * (k + max(3, args.warmup)) + 8
    st = torch.cuda.Stream(device=dev)

    def timed_model(n_layers):
        mt = synth.make_model(s, wl.wtype, args.seed + n_layers, dev, n_layers=n_layers, ctx=wl.ctx, steps=run_len)
        dec = api.Decoder(mt, max_steps=run_len, device=dev)
        with torch.cuda.stream(st):
            dec.capture(1, stream=st)
        out = []
        for _ in range(reps):
            with torch.cuda.stream(st):
                for _ in range(max(3, args.warmup)):
                    dec.replay(stream=st)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(st)
                for _ in range(k):
                    dec.replay(stream=st)
                e1.record(st)
            st.synchronize()
            out.append(e0.elapsed_time(e1) / k)
        assert api.check_device_error(st) == 0
        dec.close()
        del mt
        torch.cuda.empty_cache()
        return sorted(out)[reps // 2], out

    clocks = ClockSampler(0)
    clocks.start()
    t17, all17 = timed_model(17)
    t1, all1 = timed_model(1)
    clk = clocks.stop()
    layer_ms = (t17 - t1) / 16
    per_layer = (s.qkv_rows * s.hidden + s.hidden * s.n_q_heads * s.head_dim + 3 * s.ffn * s.hidden) * 2
    kv = s.n_kv_heads * s.head_dim * 2 * 2 * (wl.ctx + 1)
    # positions advance over the timed steps; the K/V term uses the mean position
    kv_mean = s.n_kv_heads * s.head_dim * 2 * 2 * (wl.ctx + 1 + run_len // 2)
    gbs = (per_layer + kv_mean) / (layer_ms / 1e3) / 1e9
    peak, kind = peaks()
    out = {"metric": "single-layer decode step (Qwen3-0.6B-shaped layer, position 128)",
           "value": round(1e3 / layer_ms, 1), "unit": "layer steps/s", "ms_per_layer": round(layer_ms, 5),
           "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
           "config": {"workload": wl.name, "description": wl.description,
                      "l2": "17 distinct layers (535 MB) per step, more than 4x L2; layer time = (T17 - T1) / 16",
                      "steps_each": k, "repetitions": reps},
           "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                        "frac": round(gbs / peak, 4), "peak_kind": peak_kind_label(kind),
                        "algorithmic_bytes_per_layer": int(per_layer + kv), "traffic": None},
           "repetitions": {"ms_17_layers": [round(v, 4) for v in all17], "ms_1_layer": [round(v, 4) for v in all1]},
           "clocks": clk}
    print(json.dumps(out), flush=True)


def peak_kind_label(kind):
    return f"{kind} copy peak"


def main():
    args = parse()
    if args.kernel:
        run_kernel(args)
        return
    if args.prefill:
        run_prefill_bench(args)
        return
    if args.workload == "qwen3-0.6b-layer" and args.impl != "reference":
        run_layer_bench(args)
        return
    if args.verify:
        run_verify(args)
        return
    if args.impl == "reference":
        # the oracle runs on rank 0's host cores only; other ranks exit without work
        if int(os.environ.get("RANK", "0")) == 0:
            run_reference(args, None, 0, int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0")))
        return
    dist, rank, world, local = dist_setup(args)
    try:
        if args.impl == "reference":
            run_reference(args, dist, rank, world, local)
        else:
            run_ours(args, dist, rank, world, local)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
