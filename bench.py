"""Decode benchmark of the fixed-point forward pass on GB300.

Workload: the 7B-shaped fixed-point model (dim 4096, 32 layers, 32 heads x 128, FFN hidden
11008, vocab 32000, context 2048, ~6.6 GB of int8 weights), seeded synthetic weights, a
single run: 128 prompt ids (the 127 that generate nothing prefilled layer-major), then
greedy decode.  A step is one generating position: phases 3 to 19 over all 32 layers and
the classifier.

Prints one JSON line:
  value      decode tokens/s, device-timed (CUDA events on the launching stream) over
             exactly --steps positions after --warmup untimed ones, max over ranks;
  e2e        the same metric through the public call a streaming user makes: one
             ck_turn per token with the token read back on the host every step;
  roofline   the matrix-row kernel at the decode's largest launch shape (gate and up rows
             of one layer, 22016 x 4096), timed live with CUDA events, against the measured
             HBM copy bandwidth;
  cpu_baseline  the CPU oracle on a bounded sample of the same decode (it continues from
             the GPU's state after the prefill and the first token, never past the run's
             last token), whose tokens must equal the GPU's (bitexact);
  matrow_sweep  GB/s of the matrix-row kernel on the four sweep shapes;
  prefill    the 127 prompt positions of the workload, layer-major (device-timed);
  batched_runs  the 1B-shaped model with 64 independent runs (64 prompt ids each, prefilled
             per run), generating positions of all 64 advanced together per ck_turn_batch
             pass, device-timed over --batched-passes passes;
  long_context  the 1B-shaped model at 8,192 context: 7,936 prompt ids prefilled layer-major,
             then --long-steps generating positions (~position 7,940), device-timed.
``--impl reference`` times the CPU oracle alone on the same workload, prompt and positions.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

PATHS = {"auto": 0, "step": 1, "kernels": 2}  # ck_set_path values (CK_PATH_AUTO, _STEP, _KERNELS)
METRIC = "decode tokens/s bit-exact vs oracle; matrow HBM GB/s as % of GB300 peak"
WORKLOAD = ("llama7b_shape fixed-point decode: dim 4096, 32 layers, 32 heads x 128, FFN hidden 11008, "
            "vocab 32000, context 2048, u8 weights + u32 row scales (6.61 GB/token); 128 prompt ids "
            "prefilled, then greedy decode; single run per GPU")
WORKLOAD_TOKENS = 256  # tokens a run of the workload generates
FALLBACK_HBM_GBS = 6800.0


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def matrow_bytes(rows: int, cols: int) -> int:
    """Algorithmic bytes of one matrix-row launch: each weight byte, each row scale and
    output, and the input vector read once."""
    return rows * cols + 4 * rows + 8 * rows + 8 * cols


def step_bytes(spec, pos: int) -> int:
    """Algorithmic bytes of one generating position at `pos`: every weight byte and row
    scale once, the K and V cache words of the positions 0..pos once each, the new K/V words,
    and the vectors (negligible, counted as the matrix inputs and outputs)."""
    d, h, kv, L, V = spec.dim, spec.hidden, spec.kv_dim, spec.layers, spec.vocab
    rows = L * (d + 2 * kv + d + 2 * h + d) + V
    weights = spec.weight_bytes_per_token() + 4 * rows
    kv_read = L * (pos + 1) * kv * 4 * 2
    kv_write = L * kv * 4 * 2
    vectors = 8 * (L * (4 * d + 3 * d + 2 * h + h + d) + V + d)
    return weights + kv_read + kv_write + vectors


def step_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("ck_step.cu", "ck_internal.cuh"):
        with open(os.path.join(ROOT, "fixed_point_int8_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def step_traffic(alg_per_launch: int):
    """DRAM bytes per launch of the one-position kernel: the committed ncu capture's ratio of
    traffic to algorithmic bytes (a 4-layer cut of the same model) times this launch's
    algorithmic bytes, if the capture was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "step_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("kernel_source_hash") == step_source_hash():
            return int(round(float(d["traffic_over_algorithmic"]) * alg_per_launch))
    except Exception:
        pass
    return None


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("ck_matrow.cu", "ck_internal.cuh"):
        with open(os.path.join(ROOT, "fixed_point_int8_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(shape_key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current
    kernel source; otherwise None."""
    path = os.path.join(ROOT, "profiles", "matrow_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("kernel_source_hash") == kernel_source_hash() and shape_key in d.get("launches", {}):
            return int(d["launches"][shape_key]["dram_bytes"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.seek(0)
        sm, smax, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.file:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() in ("active", "1"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- distributed plumbing

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    import torch
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- the workload

def workload_spec(args):
    import synth
    spec = synth.LLAMA7B
    if args.layers:
        import dataclasses
        spec = dataclasses.replace(spec, layers=args.layers)  # profiling and test aid only
    return spec


def workload_config(args, n_prompt: int, timed: int, parallelism: str) -> dict:
    wl = WORKLOAD if not args.layers else WORKLOAD + f" (cut to {args.layers} layers)"
    if n_prompt != 128:
        wl = wl.replace("128 prompt ids", f"{n_prompt} prompt ids")
    return {"workload": wl, "prompt_ids": n_prompt, "decode_positions_timed": timed,
            "first_timed_position": n_prompt + args.warmup,
            "l2": "inputs larger than L2: 6.6 GB of weights streamed per step",
            "parallelism": parallelism}


# ---------------------------------------------------------------- our arm

def run_ours(args):
    import torch
    import fixed_point_int8_gb300 as ck
    from fixed_point_int8_gb300 import build as libbuild
    import synth

    rank, world, local = dist_setup(args.gpus)
    libbuild.build()
    if args.batched_only:
        # profiling aid: only the 64-run batched measurement
        print(json.dumps({"batched_runs": batched_runs(ck, torch, synth, args.batched_passes, args.batched_layers)}),
              flush=True)
        return
    if args.long_only:
        # profiling aid: only the long-context measurement (optionally cut to fewer layers)
        print(json.dumps({"long_context": long_context(ck, torch, synth, args.long_steps, args.long_layers, PATHS[args.path])}),
              flush=True)
        return
    if args.matrow_only:
        # profiling aid: only the matrix-row timing of one shape, e.g. 22016x4096
        rows, cols = (int(v) for v in args.matrow_only.split("x"))
        avg, nb, alone = time_matrow(ck, torch, rows, cols, 5)
        print(json.dumps({"matrow": args.matrow_only, "us": round(avg * 1e3, 2),
                          "GB/s": round(nb / (avg * 1e-3) / 1e9, 1), "us_one_by_one": round(alone * 1e3, 2)}),
              flush=True)
        return
    spec = workload_spec(args)
    n_prompt = args.prompt_ids
    K, W = args.steps, args.warmup
    e2e_steps = min(K, args.e2e_steps)
    # the state holds the workload's whole run (256 generated tokens), or more when the
    # requested steps need them; the CPU baseline continues the same run
    max_tokens = max(WORKLOAD_TOKENS, 1 + W + K + e2e_steps)
    assert n_prompt + max_tokens - 1 <= spec.context, "too many steps for the context"

    t0 = time.time()
    art = synth.build_artifact(spec)
    ids = synth.prompt_ids(spec, n_prompt, run=rank)
    rc, model = ck.Model.load(art)
    assert rc == 0, f"ck_load_model failed: {rc}"
    path = PATHS[args.path]
    assert model.set_path(path) == 0
    state = model.new_state(n_prompt, max_tokens)
    assert model.init_state(state, ids, max_tokens) == 0
    stream = torch.cuda.current_stream()
    setup_s = time.time() - t0

    # prefill: prompt positions 0..126 layer-major, then position 127, which generates the
    # first token
    torch.cuda.synchronize()
    pev0, pev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pev0.record(stream)
    rc, res = model.turn(state, n_prompt - 1)
    pev1.record(stream)
    torch.cuda.synchronize()
    assert rc == 0 and res["work"] == n_prompt - 1, (rc, res)
    prefill_ms = pev0.elapsed_time(pev1)
    rc, res = model.turn(state, 1)
    assert rc == 0 and res["generated"] == 1, (rc, res)
    snapshot = ck.state_download(state) if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None

    # warm-up steps (untimed)
    rc, res = model.turn(state, W)
    assert rc == 0 and res["work"] == W

    sampler = ClockSampler(torch.cuda.current_device())
    with sampler:
        time.sleep(0.3)
        barrier(world)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        rc, res = model.turn(state, K)
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        assert rc == 0 and res["work"] == K, (rc, res)
        dev_ms = ev0.elapsed_time(ev1)

        # e2e: one public ck_turn call per token, its token read back on the host each step
        torch.cuda.synchronize()
        e2e_tokens = []
        t_e = time.perf_counter()
        for _ in range(e2e_steps):
            rc, r = model.turn(state, 1)
            e2e_tokens.append(r["token"])
        e2e_s = time.perf_counter() - t_e
        assert rc == 0
    clocks = sampler.summary()

    ms_max = max_over_ranks(dev_ms, world)
    value = K * world / (ms_max / 1e3)
    e2e_max = max_over_ranks(e2e_s, world)
    e2e_value = e2e_steps * world / e2e_max if e2e_steps else None

    rc, toks = model.output_tokens(state)
    assert rc == 0

    roof, sweep = matrow_measurements(ck, torch, args)
    kernel_path = "step" if args.path == "step" else "kernels"  # ck_set_path: auto takes the phase kernels
    # the whole position: weights, row scales and cache words read once, over the device time
    p0 = n_prompt + W  # first timed position
    alg = sum(step_bytes(spec, p) for p in range(p0, p0 + K))
    hbm_peak, peak_kind = load_peaks()
    achieved = alg / (dev_ms * 1e-3) / 1e9
    position_roof = {"launch": f"one decode position ({'the persistent kernel' if kernel_path == 'step' else 'all phase kernels'})",
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "peak_kind": peak_kind,
                     "algorithmic_bytes": alg // K, "ms": round(dev_ms / K, 4)}
    roof_matrow = None
    if kernel_path == "step":
        # the one-position kernel is the whole path: one launch per position
        roof_matrow = roof
        roof = {"kernel": "k_step", "launch": "one decode position (all 32 layers, classifier, maximum pass)",
                "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "peak_kind": peak_kind,
                "traffic": step_traffic(alg // K), "traffic_note": "scaled from a 4-layer ncu capture",
                "algorithmic_bytes": alg // K,
                "avg_launch_us": round(dev_ms * 1e3 / K, 2)}

    cpu = None
    bitexact = None
    if snapshot is not None:
        cpu, bitexact = cpu_baseline(art, snapshot, toks, args.cpu_seconds)
    batched = None
    longc = None
    if (args.batched_passes or args.long_steps) and rank == 0:
        del model, state
        torch.cuda.empty_cache()
        if args.batched_passes:
            batched = batched_runs(ck, torch, synth, args.batched_passes, args.batched_layers)
            torch.cuda.empty_cache()
        if args.long_steps:
            longc = long_context(ck, torch, synth, args.long_steps, args.long_layers, path)

    if rank != 0:
        return
    # our kernels per position: the one-position kernel, or embedding + five per layer
    # (four matrix-row launches and attention) + classifier + maximum pass
    launches_per_step = 1 if kernel_path == "step" else 1 + 5 * spec.layers + 2
    weight_bytes = spec.weight_bytes_per_token()
    hbm, peak_kind = load_peaks()
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(ms_max / K, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u8 x i64 (int64 activations, 16 fractional bits)",
        "data": "synthetic (seeded weights and prompt ids, no checkpoint)",
        "config": workload_config(args, n_prompt, K, "replicas" if world > 1 else "single GPU"),
        "roofline": roof,
        "weight_roofline": {"bytes_per_token": weight_bytes,
                            "tokens_per_s_at_peak": round(hbm * 1e9 / weight_bytes, 1),
                            "frac": round(value / world / (hbm * 1e9 / weight_bytes), 4),
                            "peak_gbs": hbm, "peak_kind": peak_kind},
        "e2e": {"value": round(e2e_value, 2) if e2e_value else None, "unit": "tokens/s",
                "h2d_bytes_per_step": 8, "d2h_bytes_per_step": 512,
                "how": "ck_turn(1 position) per token; the call reads the 256-byte state header "
                       "before and after and writes the 8-byte turn counter"},
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "bitexact": bitexact,
        "matrow_sweep": sweep,
        "matrow_roofline": roof_matrow,
        "position_roofline": position_roof,
        "prefill": {"value": round((n_prompt - 1) / (prefill_ms * 1e-3), 1), "unit": "prompt positions/s",
                    "positions": n_prompt - 1, "ms": round(prefill_ms, 3),
                    "how": "one ck_turn over the prompt positions that generate no token: layer-major "
                           "chunks, byte-plane f16 MMA contraction (CUDA events on the stream)"},
        "batched_runs": batched,
        "long_context": longc,
        "path": kernel_path,
        "setup_s": round(setup_s, 1),
    }
    print(json.dumps(line), flush=True)


def batched_runs(ck, torch, synth, passes, layers=0):
    """The 1B-shaped model with 64 runs: each prefilled per run, then `passes` generating
    passes of ck_turn_batch (one position of every run each), device-timed after three
    untimed passes.  `layers` cuts the model (a test aid; 0: the whole model)."""
    import dataclasses
    wl = synth.WORKLOADS["1b_x64"]
    spec = wl.spec if not layers else dataclasses.replace(wl.spec, layers=layers)
    passes = min(passes, wl.steps - 4)
    rc, m = ck.Model.load(synth.build_artifact(spec))
    assert rc == 0
    states = []
    for r in range(wl.runs):
        sg = m.new_state(wl.n_prompt, wl.steps)
        assert m.init_state(sg, synth.prompt_ids(spec, wl.n_prompt, run=r), wl.steps) == 0
        assert m.turn(sg, wl.n_prompt - 1)[0] == 0
        states.append(sg)
    for _ in range(3):
        rc, res, rcs = m.turn_batch(states)
        assert rc == 0
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(passes):
        rc, res, rcs = m.turn_batch(states)
        assert rc == 0 and all(x["generated_this_turn"] == 1 for x in res)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    value = wl.runs * passes / (ms * 1e-3)
    macs = spec.weight_bytes_per_token() * wl.runs  # one u8 x i64 multiply-add per weight and run
    peak = None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak = float(json.load(f)["bf16_tflops"])
    except Exception:
        pass
    tflops = 2 * macs / (ms * 1e-3 / passes) / 1e12
    return {"value": round(value, 1), "unit": "tokens/s", "runs": wl.runs, "passes": passes,
            "ms_per_pass": round(ms / passes, 3),
            "workload": f"1b_shape (dim 2048, {spec.layers} layers, 32 heads, FFN 5632, vocab 32000), 64 runs "
                        f"x 64 prompt ids, positions 67.. of each run, greedy",
            "algorithmic_tflops": round(tflops, 1),
            "algorithmic_frac_of_bf16_peak": round(tflops / peak, 4) if peak else None,
            "note": "whole pass (all kernels); algorithmic = 2 x weights x runs per pass, the byte "
                    "planes multiply the tensor work by the plane count (3 here)"}


def long_context(ck, torch, synth, steps, layers, path=0):
    """The 1B-shaped model at 8,192 context: 7,936 prompt ids prefilled layer-major (one
    ck_turn), then `steps` generating positions in one ck_turn, both device-timed; `path`
    is the ck_set_path choice for the generating positions."""
    import dataclasses
    wl = synth.WORKLOADS["1b_long"]
    spec = wl.spec if not layers else dataclasses.replace(wl.spec, layers=layers)
    steps = max(1, min(steps, wl.steps - 4))
    rc, m = ck.Model.load(synth.build_artifact(spec))
    assert rc == 0
    assert m.set_path(path) == 0
    st = m.new_state(wl.n_prompt, wl.steps)
    assert m.init_state(st, synth.prompt_ids(spec, wl.n_prompt), wl.steps) == 0
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    torch.cuda.synchronize()
    ev[0].record(stream)
    rc, res = m.turn(st, wl.n_prompt - 1)
    ev[1].record(stream)
    assert rc == 0 and res["work"] == wl.n_prompt - 1
    rc, res = m.turn(st, 3)  # the first generating positions, untimed
    assert rc == 0
    ev[2].record(stream)
    rc, res = m.turn(st, steps)
    ev[3].record(stream)
    torch.cuda.synchronize()
    assert rc == 0 and res["work"] == steps
    pre_ms, dec_ms = ev[0].elapsed_time(ev[1]), ev[2].elapsed_time(ev[3])
    pos = wl.n_prompt + 2
    kv = spec.layers * (pos + steps // 2 + 1) * spec.kv_dim * 4 * 2
    per_token = spec.weight_bytes_per_token() + kv
    return {"decode": {"value": round(steps / (dec_ms * 1e-3), 1), "unit": "tokens/s",
                       "positions": f"{pos}..{pos + steps - 1}",
                       "bytes_per_token": per_token,
                       "achieved_gbs": round(per_token / (dec_ms * 1e-3 / steps) / 1e9, 1)},
            "prefill": {"value": round((wl.n_prompt - 1) / (pre_ms * 1e-3), 1), "unit": "prompt positions/s",
                        "positions": wl.n_prompt - 1, "ms": round(pre_ms, 1)},
            "workload": f"1b_shape{' cut to %d layers' % layers if layers else ''}, context 8192, "
                        f"{wl.n_prompt} prompt ids, greedy"}


def time_matrow(ck, torch, rows, cols, iters):
    """Average duration (ms) of ck_matrow launches of one shape.  The launches run back to back
    on the current stream between one pair of CUDA events, queued behind a device-side wait so
    that host-side call overhead never leaves the GPU idle inside the timed region; the matrix
    rotates through copies totalling three times the L2 size so every launch streams from HBM.
    Also returns the average of the same launches timed one by one (an event pair around each).
    Returns (ms back to back, algorithmic bytes, ms one by one)."""
    import synth
    stream = torch.cuda.current_stream()
    l2 = getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 128 << 20)
    W, s, x = synth.matrow_case(rows, cols)
    nbytes = rows * cols
    copies = max(2, -(-3 * l2 // nbytes))
    Wd = torch.from_numpy(W).cuda()
    Ws = [Wd] + [Wd.clone() for _ in range(copies - 1)]
    sd = torch.from_numpy(s.view(np.int32)).cuda()
    xd = torch.from_numpy(x).cuda()
    y = torch.empty(rows, dtype=torch.int64, device="cuda")
    for i in range(3):
        rc, _ = ck.matrow(Ws[i % copies], sd, xd, out=y)
        assert rc == 0
    torch.cuda.synchronize()
    torch.cuda._sleep(4_000_000)  # about 2 ms of device time while the host queues the launches
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(iters):
        ck.matrow(Ws[i % copies], sd, xd, out=y)
    b.record(stream)
    torch.cuda.synchronize()
    ms_run = a.elapsed_time(b) / iters
    times = []
    for i in range(iters):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        ck.matrow(Ws[i % copies], sd, xd, out=y)
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    ms_alone = sum(a.elapsed_time(b) for a, b in times) / iters
    del Ws, Wd
    torch.cuda.empty_cache()
    return ms_run, matrow_bytes(rows, cols), ms_alone


def matrow_measurements(ck, torch, args):
    """Times ck_matrow launches with CUDA events on the current stream, back to back (the
    reported figure) and one by one (context: each then also pays the launch and event
    latency); matrices rotate through copies whose total exceeds the L2 cache so every
    launch streams from HBM."""
    import synth
    hbm, peak_kind = load_peaks()
    sweep = {}
    for rows, cols in synth.MATROW_SHAPES:
        avg, nb, alone = time_matrow(ck, torch, rows, cols, 30)
        gbs = nb / (avg * 1e-3) / 1e9
        sweep[f"{rows}x{cols}"] = {"us": round(avg * 1e3, 2), "GB/s": round(gbs, 1),
                                   "frac_of_peak": round(gbs / hbm, 4), "us_one_by_one": round(alone * 1e3, 2)}
    rows, cols = 2 * 11008, 4096
    avg, nb, alone = time_matrow(ck, torch, rows, cols, 30)
    achieved = nb / (avg * 1e-3) / 1e9
    key = f"{rows}x{cols}"
    traffic = ncu_traffic(key)
    roof = {"kernel": "k_matrow", "launch": f"{key} (gate and up rows of one 7B layer)",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(achieved / hbm, 4), "peak_kind": peak_kind,
            "traffic": traffic, "algorithmic_bytes": nb, "avg_launch_us": round(avg * 1e3, 2),
            "timing": "30 launches back to back between one event pair",
            "avg_launch_us_one_by_one": round(alone * 1e3, 2)}
    return roof, sweep


def cpu_baseline(art, snapshot, gpu_tokens, budget_s):
    """The oracle, as it stands, continues the decode from the GPU's state after the prefill
    for as many positions as fit in about budget_s seconds, never past the run's last token
    (the state's max tokens); its tokens must equal the GPU's."""
    import oracle
    m = oracle.Model(art)
    st = snapshot.copy()
    h = oracle.header(st)
    start = h["generated"]
    room = min(h["max_tokens"] - start, len(gpu_tokens) - start)
    t0 = time.perf_counter()
    n, rc, el = 0, 0, 0.0
    while n < room:
        rc, res = m.turn(st, 1)
        el = time.perf_counter() - t0
        if rc != 0 or res["generated_this_turn"] != 1:
            break
        n += 1
        if el > budget_s:
            break
    if n == 0:
        return None, {"checked_tokens": start, "equal": False, "oracle_rc": rc}
    lay = m.layout(h["n_prompt"], h["max_tokens"])
    otoks = st[lay["out"]:lay["out"] + 4 * (start + n)].view("<u4").tolist()
    same = otoks == list(gpu_tokens[:start + n])
    cpu = {"value": round(n / el, 4), "unit": "tokens/s", "cores": oracle.threads(), "kind": "oracle",
           "sample": f"{n} decode positions of the same 7B-shaped run, continued on the CPU from the "
                     f"GPU's state after the prefill and the first token (OpenMP over independent matrix "
                     f"rows)"}
    return cpu, {"checked_tokens": start + n, "equal": bool(same), "oracle_rc": rc}


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    """The CPU oracle as the reference implementation of the same decode, on rank 0 only:
    it runs the workload's prompt ids (the positions that generate nothing, then the one
    that generates the first token), --warmup generating positions untimed, then times up
    to --steps generating positions, the same positions the GPU arm times, stopping early
    after --reference-seconds."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    import synth
    spec = workload_spec(args)
    art = synth.build_artifact(spec)
    m = oracle.Model(art)
    K, W = args.steps, args.warmup
    n_prompt = args.prompt_ids
    max_tokens = max(WORKLOAD_TOKENS, 1 + W + K)
    rc, st = m.init_state(synth.prompt_ids(spec, n_prompt), max_tokens)
    assert rc == 0
    t_pre = time.perf_counter()
    rc, res = m.turn(st, n_prompt)  # the prompt positions and the first generated token
    pre_s = time.perf_counter() - t_pre
    assert rc == 0 and res["generated"] == 1, (rc, res)
    rc, _ = m.turn(st, W)
    assert rc == 0
    t0 = time.perf_counter()
    done = 0
    for _ in range(K):
        rc, _ = m.turn(st, 1)
        assert rc == 0
        done += 1
        if time.perf_counter() - t0 > args.reference_seconds:
            break
    el = time.perf_counter() - t0
    value = done / el
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": done, "steps_requested": K,
        "warmup": W, "ms_per_step": round(el / max(done, 1) * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8 x i64 (int64 activations, 16 fractional bits)",
        "data": "synthetic (seeded weights and prompt ids, no checkpoint)",
        "config": workload_config(args, n_prompt, done, "CPU oracle"),
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": oracle.threads(), "kind": "oracle",
                         "sample": f"generating positions {n_prompt + W}..{n_prompt + W + done - 1} of the "
                                   f"workload's run ({done} timed after {W} warm-up positions; the "
                                   f"{n_prompt} prompt positions took {pre_s:.1f} s, untimed)"},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=253)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=64)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--reference-seconds", type=float, default=150.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batched-passes", type=int, default=40,
                    help="passes of the 64-run batched measurement (0: skip it)")
    ap.add_argument("--batched-only", action="store_true",
                    help="profiling aid: run only the 64-run batched measurement")
    ap.add_argument("--batched-layers", type=int, default=0,
                    help="test aid: cut the 64-run model to this many layers")
    ap.add_argument("--long-steps", type=int, default=40,
                    help="generating positions of the 8K-context measurement (0: skip it)")
    ap.add_argument("--long-only", action="store_true",
                    help="profiling aid: run only the 8K-context measurement")
    ap.add_argument("--long-layers", type=int, default=0,
                    help="profiling aid: cut the 8K-context model to this many layers")
    ap.add_argument("--path", choices=("auto", "step", "kernels"), default="auto",
                    help="one persistent kernel per position (step) or one kernel per phase")
    ap.add_argument("--prompt-ids", type=int, default=128,
                    help="prompt length (the workload uses 128; shorter only for profiling)")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling aid: the same model with fewer layers (small ncu captures)")
    ap.add_argument("--matrow-only", default="",
                    help="profiling aid: time ck_matrow on one ROWSxCOLS shape and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
