"""Throughput of UniPrefill's per-layer drop step on GB300, through the C ABI.

One step = one pass of the whole hot path over one batch:
  up_score_blocks (Eqs. 2-4) -> up_select_topp (Eq. 5/14) -> up_compact (+ metadata, history)
  -> up_slot_mapping (Eq. 16, next layer) -> up_scatter_back (Eq. 8) -> up_seqused (Eq. 17)
value = tokens of the batch / device time of one step (CUDA events on the launching stream).

Default workload: a Gemma-3-12B-shaped full-attention layer under load, 64 requests of 32768 tokens
packed (2,097,152 tokens; 16/8 heads, d_k 256, hidden 3840, G 64, n 128, A 128, p 0.99), the
largest workload that fits one GPU, with seeded synthetic bf16 inputs.  The same line carries, under
"per_config", the other four workloads measured the same way (one 4K and one 32K LLaMA-3.1-8B-shaped
request, 16 log-uniform requests of 4K-128K, four Qwen3-Next-shaped 128K requests).  L2 is
flushed (512 MB write) before every timed step.  `--impl reference` times the fp64 CPU oracle
on the host cores instead (bounded sample of the same workload per step).  `--sweep rho|ablation`
prints measured sweeps instead of the step line (compaction against the kept fraction; the stages
over G, n and p); `--sweep stack` times a random-weight decoder stack with one drop against the top-p
threshold (the saving of Eqs. 7-10).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill tokens/s through score+top-p+compact; % of tensor/HBM roofline"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", type=int, default=5,
                    help="workload index 1..5 (default 5: Gemma-3-12B layer geometry, 64 x 32K, the largest)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other four workloads' measurement (the 'per_config' object of the line)")
    ap.add_argument("--per-config-steps", type=int, default=100)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--p", type=float, default=None, help="override the workload's top-p threshold")
    ap.add_argument("--requests", type=int, default=None,
                    help="keep only the workload's first K requests (a smaller case of the same geometry)")
    ap.add_argument("--sweep", choices=["rho", "ablation", "stack"], default=None,
                    help="instead of the step line, one JSON line per point: 'rho' = compaction and scatter "
                         "bandwidth against the kept fraction; 'ablation' = the step's stages over G, n and p; "
                         "'stack' = a random-weight decoder stack with one drop, against the top-p threshold")
    ap.add_argument("--stack-layers", type=int, default=32, help="layers of the --sweep stack decoder stack")
    ap.add_argument("--drop-layer", type=int, default=10, help="0-based layer of the --sweep stack drop")
    ap.add_argument("--stack-ffn", type=int, default=14336, help="FFN width of the --sweep stack layers")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clocks and throttle reasons while the GPU is under load."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0, period_ms=20):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", f"-lms={period_ms}"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 7:
                continue
            try:
                rows.append((ts, float(parts[0]), float(parts[1]), parts[3:]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median([r[1] for r in inside]) if inside else None,
                "sm_max_mhz": max([r[2] for r in inside]) if inside else None,
                "reasons": reasons, "samples": len(inside)}


# ------------------------------------------------------------------------------------------ our arm

def run_gb300(args, w, rank, world, steps=None, sample_clocks=True):
    import torch
    import long_context_prefill_varlen_gb300 as up
    from synth import cpu as gen
    from synth import gpu as sgpu

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    up.load_library()
    stream = torch.cuda.current_stream()

    inputs = sgpu.build_device(w, device=dev)
    cu = inputs["cu_seqlens"]
    L, layer, B = 4, 1, 16
    step = up.DropStep(cu, w.T, w.Hq, w.Hkv, w.dk, w.hdim, G=w.G, n=w.n, A=w.A, p=w.p, L=L, layer=layer,
                       device=dev)
    mb = max(1, max(-(-N // B) for N in w.lengths))
    rng = np.random.default_rng(12345)
    table = torch.from_numpy(rng.permutation(w.R * mb).reshape(w.R, mb).astype(np.int32)).to(dev)
    next_slots = torch.empty(max(1, w.T), dtype=torch.int64, device=dev)
    residual = inputs["hidden"].clone()
    orig_len = torch.tensor(w.lengths, dtype=torch.int32, device=dev)
    kv_len = orig_len.clone()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def run_step(marks=None):
        def mark(i):
            if marks is not None:
                marks[i].record(stream)
        mark(0)
        step.score(inputs["Q"], inputs["K"])
        mark(1)
        step.select()
        mark(2)
        step.compact(inputs["hidden"], inputs["positions"], inputs["slots"])
        mark(3)
        up.up_slot_mapping(step.out_positions[:w.T], step.new_cu, table, B, next_slots, step.status,
                           num_tokens=step.num_actual)
        mark(4)
        step.scatter_back(step.out_hidden, residual)
        mark(5)
        step.seqused(orig_len, kv_len, layer + 1)
        mark(6)

    for _ in range(max(3, args.warmup)):
        flush.fill_(1)
        run_step()
    torch.cuda.synchronize()
    step.check()
    kept = int(step.num_actual.item())

    # Kernels one step launches (counted by the library on the eager path; a graph replay launches the same).
    l0 = up.up_kernel_launches()
    run_step()
    torch.cuda.synchronize()
    per_step = up.up_kernel_launches() - l0

    # The step captured once as a CUDA graph; the timed region replays it, one event pair per step on
    # the stream the graph is launched on, the L2 flush outside the pair.
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        run_step()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run_step()
    torch.cuda.synchronize()
    for _ in range(3):
        flush.fill_(1)
        graph.replay()
    torch.cuda.synchronize()

    steps = args.steps if steps is None else steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sampler = ClockSampler(dev.index) if rank == 0 and sample_clocks else None
    time.sleep(0.3 if sampler else 0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(steps):
        flush.fill_(1)                      # L2 flush, outside the event pair
        ev[k][0].record(stream)
        graph.replay()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    launches = per_step * steps
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop(t0, t1) if sampler else None
    step.check()
    step_ms = np.array([a.elapsed_time(b) for a, b in ev])
    ms = float(step_ms.mean())
    spread = {"median": float(np.median(step_ms)), "p10": float(np.percentile(step_ms, 10)),
              "p90": float(np.percentile(step_ms, 90)), "max": float(step_ms.max())}
    if world > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())

    # Per-stage breakdown (eager launches, an event between stages, L2 flushed before each step): it
    # attributes the step's time; each stage's share includes its own launch gaps.
    nst = 7
    nb = min(steps, 100)
    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(nst)] for _ in range(nb)]
    torch.cuda.synchronize()
    for k in range(nb):
        flush.fill_(1)
        run_step(marks[k])
    torch.cuda.synchronize()
    step.check()
    stage_ms = np.zeros((nb, nst - 1))
    for k in range(nb):
        for i in range(nst - 1):
            stage_ms[k, i] = marks[k][i].elapsed_time(marks[k][i + 1])
    del graph
    return dict(ms=ms, spread=spread, eager_ms=float(stage_ms.sum(axis=1).mean()), stage_ms=stage_ms.mean(axis=0),
                launches=launches, per_step_launches=per_step, clocks=clocks, kept=kept,
                kstar=step.kstar.cpu().tolist(), near_threshold=near_threshold_blocks(w, step), step=step,
                inputs=inputs, run_step=run_step, dev=dev,
                flush=flush, geometry=dict(L=L, layer=layer, B=B, table=table, orig_len=orig_len, kv_len=kv_len))


def near_threshold_blocks(w, step, rtol=1e-3):
    """Blocks, other than each request's k*-th ranked block, whose score lies within rtol (relative) of
    that block's score tau, from the GPU's own block scores: the only blocks whose keep decision the
    parity tolerance lets differ from the oracle's (the parity tests count the actual differences)."""
    bs = step.block_scores.cpu().numpy().astype(np.float64)
    ks = step.kstar.cpu().numpy()
    cu = w.cu_seqlens()
    b0, count = 0, 0
    for r in range(w.R):
        nb = -(-(cu[r + 1] - cu[r]) // w.G)
        if nb and ks[r] > 0:
            b = bs[b0:b0 + nb]
            order = np.lexsort((-np.arange(nb), -b))         # descending score, then higher index first
            tau = b[order[ks[r] - 1]]
            count += int((np.abs(b - tau) <= rtol * tau).sum()) - 1
        b0 += nb
    return count


def e2e_measure(args, w, ctx):
    """The step through the C ABI with the batch in pinned HOST memory, step after step with two in
    flight: step k+1's inputs go host -> device on one copy stream while step k's result comes back on
    another (the link moves both directions at once), each step on its own device buffer set, reused
    two steps later.  Every step's H2D of the inputs the calls read and D2H of its result (the compacted
    hidden / positions / slots at their upper bound T rows, so the host never waits for T', and the new
    metadata) is inside the timed region."""
    import torch
    import long_context_prefill_varlen_gb300 as up
    dev, g = ctx["dev"], ctx["geometry"]
    pin = {k: ctx["inputs"][k].cpu().pin_memory() for k in ("K", "hidden", "positions", "slots")}
    Qh = ctx["inputs"]["Q"].cpu().pin_memory()
    cu = w.cu_seqlens()
    wins = [(max(cu[r], cu[r + 1] - w.n), cu[r + 1]) for r in range(w.R)]     # the query rows the score reads
    h2d = sum(t.numel() * t.element_size() for t in pin.values()) + sum((b - a) * w.Hq * w.dk * 2 for a, b in wins)
    sets = []
    for i in range(2):
        inp = ctx["inputs"] if i == 0 else {k: (torch.empty_like(v) if torch.is_tensor(v) else v)
                                            for k, v in ctx["inputs"].items()}
        if i:
            inp["cu_seqlens"].copy_(ctx["inputs"]["cu_seqlens"])
        st = ctx["step"] if i == 0 else up.DropStep(inp["cu_seqlens"], w.T, w.Hq, w.Hkv, w.dk, w.hdim, G=w.G,
                                                    n=w.n, A=w.A, p=w.p, L=g["L"], layer=g["layer"], device=dev)
        out = dict(hidden=torch.empty(w.T, w.hdim, dtype=torch.bfloat16).pin_memory(),
                   positions=torch.empty(w.T, dtype=torch.int64).pin_memory(),
                   slots=torch.empty(w.T, dtype=torch.int64).pin_memory(),
                   meta=torch.empty(w.R + 2, dtype=torch.int32).pin_memory())
        sets.append(dict(inp=inp, step=st, out=out, residual=torch.empty_like(inp["hidden"]),
                         next_slots=torch.empty(max(1, w.T), dtype=torch.int64, device=dev),
                         seq=torch.zeros(w.R, dtype=torch.int32, device=dev)))
    d2h = w.T * (w.hdim * 2 + 16) + (w.R + 2) * 4
    s_in, s_run, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = [dict(inp=torch.cuda.Event(), run=torch.cuda.Event(), out=torch.cuda.Event()) for _ in range(2)]

    def issue(k):
        S, E = sets[k % 2], ev[k % 2]
        inp, st = S["inp"], S["step"]
        with torch.cuda.stream(s_in):
            s_in.wait_event(E["run"])                     # the set's previous step has read its inputs
            for name in pin:
                inp[name].copy_(pin[name], non_blocking=True)
            for a, b in wins:
                inp["Q"][a:b].copy_(Qh[a:b], non_blocking=True)
            E["inp"].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(E["inp"])
            s_run.wait_event(E["out"])                    # and its previous result has left the device
            st.score(inp["Q"], inp["K"])
            st.select()
            st.compact(inp["hidden"], inp["positions"], inp["slots"])
            up.up_slot_mapping(st.out_positions[:w.T], st.new_cu, g["table"], g["B"], S["next_slots"], st.status,
                               num_tokens=st.num_actual)
            st.scatter_back(st.out_hidden, S["residual"])
            st.seqused(g["orig_len"], g["kv_len"], g["layer"] + 1)
            E["run"].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(E["run"])
            o = S["out"]
            o["hidden"].copy_(st.out_hidden, non_blocking=True)
            o["positions"].copy_(st.out_positions[:w.T], non_blocking=True)
            o["slots"].copy_(st.out_slots[:w.T], non_blocking=True)
            o["meta"][:w.R + 1].copy_(st.new_cu, non_blocking=True)
            o["meta"][w.R + 1:].copy_(st.num_actual, non_blocking=True)
            E["out"].record(s_out)

    for k in range(2):                                    # warm-up (both buffer sets)
        issue(k)
    torch.cuda.synchronize()
    steps = max(4, args.e2e_steps * 2)
    t0 = time.perf_counter()
    for k in range(steps):
        issue(k)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    for S in sets:
        S["step"].check()
        assert int(S["out"]["meta"][w.R + 1]) == int(S["step"].num_actual.item())
    sec = (t1 - t0) / steps
    return {"value": w.T / sec, "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": sec * 1e3, "steps": steps, "in_flight": 2,
            "note": "pinned host buffers; H2D of step k+1 overlaps D2H of step k on separate copy streams"}


# ------------------------------------------------------------------------------------------ oracle timing

def oracle_sample(w, sample_tokens):
    """Inputs of a bounded sample: one request of `sample_tokens` tokens with the workload's geometry
    (the workload itself when it is a single request of that length)."""
    from synth import cpu as gen
    if w.R == 1 and w.T == sample_tokens:
        ws = w
    else:
        ws = w.replace(lengths=(int(sample_tokens),), salt=w.index * 7 + 1)
    host = gen.materialize(ws)
    Q = gen.bf16_bits_to_f32(host["Q"]).astype(np.float64)
    K = gen.bf16_bits_to_f32(host["K"]).astype(np.float64)
    return ws, host, Q, K


def oracle_once(ws, host, Q, K):
    import oracle
    t0 = time.perf_counter()
    out = oracle.drop_step(Q, K, host["cu_seqlens"], ws.G, ws.n, ws.A, ws.p, host["hidden"],
                           host["positions"], host["slots"])
    c = out["compact"]
    oracle.carry_forward(host["hidden"], c["hidden"], c["kept_index"])
    return time.perf_counter() - t0


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, w, rank, world):
    if rank != 0:
        return None
    sample = min(w.T, 4096)
    sw = oracle_sample(w, sample)
    for _ in range(args.warmup):
        oracle_once(*sw)
    times = [oracle_once(*sw) for _ in range(args.steps)]
    sec = statistics.mean(times)
    val = sample / sec
    cores = cpu_cores()
    return {"metric": METRIC, "value": val, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w),
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"one request of {sample} tokens with the workload's geometry per step "
                                       "(score+select+compact+scatter; the per-token work does not depend on N)"},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------------------------------ sweeps

def _time_events(fn, steps, flush, stream):
    """mean device time (ms) of fn() over `steps` calls, L2 flushed before each, events on `stream`"""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for k in range(steps):
        flush.fill_(1)
        ev[k][0].record(stream)
        fn()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    return float(np.mean([a.elapsed_time(b) for a, b in ev]))


def run_sweep(args, w):
    """Measured sweeps on the workload's geometry; one JSON line per point (not the step line)."""
    import torch
    import long_context_prefill_varlen_gb300 as up
    from synth import gpu as sgpu
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    up.load_library()
    stream = torch.cuda.current_stream()
    pk, pk_kind = peaks()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    steps = max(3, min(args.steps, 50))
    if args.sweep == "rho":
        # compaction gather and scatter-back against the kept fraction: whole G-token blocks kept with
        # probability rho (seeded), the rest of the step not involved
        inputs = sgpu.build_device(w, device=dev, parts=("hidden", "positions", "slots"))
        cu = torch.tensor(w.cu_seqlens(), dtype=torch.int32, device=dev)
        step = up.DropStep(cu, w.T, w.Hq, w.Hkv, w.dk, w.hdim, G=w.G, n=w.n, A=w.A, p=w.p, device=dev)
        residual = inputs["hidden"].clone()
        rng = np.random.default_rng(7)
        nblk = -(-w.T // w.G)
        for rho in (0.1, 0.25, 0.5, 0.75, 0.9, 0.99, 1.0):
            blk = rng.random(nblk) < rho
            keep = np.repeat(blk, w.G)[:w.T].astype(np.uint8)
            step.token_keep.copy_(torch.from_numpy(keep).to(dev))
            comp = lambda: step.compact(inputs["hidden"], inputs["positions"], inputs["slots"])
            scat = lambda: step.scatter_back(step.out_hidden, residual)
            for _ in range(3):
                comp()
                scat()
            torch.cuda.synchronize()
            step.check()
            kept = int(step.num_actual.item())
            cms = _time_events(comp, steps, flush, stream)
            sms = _time_events(scat, steps, flush, stream)
            rows = 2 * kept * w.hdim * 2 + kept * 4
            print(json.dumps({"sweep": "rho", "workload": w.name, "rho": kept / w.T, "kept_tokens": kept,
                              "compact_ms": cms, "compact_gbs": rows / (cms * 1e-3) / 1e9,
                              "compact_frac_of_hbm": rows / (cms * 1e-3) / 1e9 / pk["hbm_gbs"],
                              "scatter_ms": sms, "scatter_gbs": rows / (sms * 1e-3) / 1e9,
                              "scatter_frac_of_hbm": rows / (sms * 1e-3) / 1e9 / pk["hbm_gbs"],
                              "steps": steps, "peak_source": pk_kind}), flush=True)
        return
    if args.sweep == "stack":
        run_stack_sweep(args, w, dev, stream, pk, pk_kind)
        return
    # ablation: G, n and p on the workload's geometry (the step's stages, eager, events between)
    inputs = sgpu.build_device(w, device=dev)
    cu = inputs["cu_seqlens"]
    for G in (32, 64, 128):
        for n in (32, 128, 512):
            for p in (0.98, 0.99):
                step = up.DropStep(cu, w.T, w.Hq, w.Hkv, w.dk, w.hdim, G=G, n=n, A=w.A, p=p, device=dev)
                fns = [lambda: step.score(inputs["Q"], inputs["K"]), step.select,
                       lambda: step.compact(inputs["hidden"], inputs["positions"], inputs["slots"])]
                for _ in range(3):
                    for f in fns:
                        f()
                torch.cuda.synchronize()
                step.check()
                ms = [_time_events(f, steps, flush, stream) for f in fns]
                kept = int(step.num_actual.item())
                wv = w.replace(G=G, n=n, p=p)
                print(json.dumps({"sweep": "ablation", "workload": w.name, "G": G, "n": n, "p": p,
                                  "rho": kept / w.T, "kstar": step.kstar.cpu().tolist()[:4],
                                  "score_ms": ms[0], "select_ms": ms[1], "compact_ms": ms[2],
                                  "score_frac_of_bf16_peak": score_flops(wv) / (ms[0] * 1e-3) / 1e12 / pk["bf16_tflops"],
                                  "select_share": ms[1] / sum(ms), "steps": steps}), flush=True)
                del step
                torch.cuda.empty_cache()


def run_stack_sweep(args, w, dev, stream, pk, pk_kind):
    """The saving a drop buys on a decoder stack (Eqs. 7-10): an L-layer random-weight stack of the
    workload's layer geometry over the workload's hidden states, without a drop and with one drop at
    --drop-layer for several top-p thresholds; the forward's device time against the FLOPs accounting.
    Every forward reads its weights (hundreds of MB per layer) from HBM, far beyond L2."""
    import torch
    from long_context_prefill_varlen_gb300 import layerstack as ls
    from synth import gpu as sgpu
    inputs = sgpu.build_device(w, device=dev, parts=("hidden", "positions"))
    cu = inputs["cu_seqlens"]
    g = ls.StackGeometry(d=w.hdim, Hq=w.Hq, Hkv=w.Hkv, dk=w.dk, ffn=args.stack_ffn)
    L, l1 = args.stack_layers, args.drop_layer
    stack = ls.RandomLlamaStack(L, g, seed=0, device=dev)
    max_len = max(w.lengths)
    steps = max(2, min(args.steps, 5))
    base_ms = base_fl = None
    for p in (None, 0.99, 0.95, 0.9, 0.75, 0.5):
        drops = [] if p is None else [(l1, p)]
        fwd = lambda: stack.forward(inputs["hidden"], inputs["positions"], cu, max_len, drops=drops, G=w.G, n=w.n,
                                    A=w.A)
        _, info = fwd()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in ev:
            a.record(stream)
            fwd()
            b.record(stream)
        torch.cuda.synchronize()
        ms = float(np.median([a.elapsed_time(b) for a, b in ev]))
        kept = [int(x) for x in info[0]["step"].new_len.cpu().tolist()] if info else list(w.lengths)
        fl = ls.stack_flops(w.lengths, g, L, [(l1, kept)] if info else [])
        if p is None:
            base_ms, base_fl = ms, fl
        rec = {"sweep": "stack", "workload": w.name, "layers": L, "drop_layer": None if p is None else l1, "p": p,
               "rho": sum(kept) / w.T, "ms_per_forward": ms, "prefill_tokens_per_s": w.T / (ms * 1e-3),
               "speedup_vs_no_drop": base_ms / ms, "flops_ratio_no_drop_over_this": base_fl / fl,
               "stack_tflops": fl / (ms * 1e-3) / 1e12,
               "stack_frac_of_bf16_peak": fl / (ms * 1e-3) / 1e12 / pk["bf16_tflops_sustained"],
               "steps": steps, "layers_are": "cuBLAS GEMMs + PyTorch varlen flash attention (random weights)",
               "peak": "bf16_tflops_sustained", "peak_source": pk_kind}
        print(json.dumps(rec), flush=True)
        del info
        torch.cuda.empty_cache()


# ------------------------------------------------------------------------------------------ report

def workload_config(w):
    return {"workload": w.name, "R": w.R, "T": w.T, "Hq": w.Hq, "Hkv": w.Hkv, "d_k": w.dk, "hidden": w.hdim,
            "G": w.G, "n": w.n, "A": w.A, "p": w.p, "seed": w.seed, "l2": "flushed (512 MB write) before each step",
            "timing": "the step captured as one CUDA graph, CUDA events around each replay",
            "parallelism": "request-sharded replicas, no collective on the data path"}


def source_digest(path):
    import hashlib
    with open(os.path.join(ROOT, path), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def measured_traffic(kernel, w):
    """DRAM bytes per launch from the committed ncu summary, or None if the kernel changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel, {}).get(f"config{w.index}")
    if not e or e.get("source_sha256_16") != source_digest(e["source"]):
        return None
    return e["dram_bytes_per_launch"]


def score_input_bytes(w):
    """DRAM input of the score call: K once, plus the window rows of Q once per (KV head) unit."""
    kb = w.T * w.Hkv * w.dk * 2
    qb = sum(min(w.n, N) for N in w.lengths) * w.Hq * w.dk * 2
    return kb + qb


def score_flops(w):
    """Algorithmic FLOPs of the score call: S = Q K^T over the causal support once,
    2 * d_k * (n_eff*N - n_eff(n_eff-1)/2) per (request, query head).  The call computes S once (the
    one-pass form; a second pass over the block sums replaces the recompute of S)."""
    tot = 0
    for N in w.lengths:
        ne = min(w.n, N)
        tot += 2 * w.dk * (ne * N - ne * (ne - 1) // 2) * w.Hq
    return tot


def main():
    args = parse()
    rank, world = int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))
    if world > 1:
        import torch
        import torch.distributed as dist
        if args.impl == "reference":
            dist.init_process_group("gloo")
        else:
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
            dist.init_process_group("nccl")
    from synth import recipe
    w = recipe.workload(args.config)
    if args.p is not None:
        w = w.replace(p=args.p)
    if args.requests is not None and args.requests < w.R:
        k = max(1, args.requests)
        w = w.replace(lengths=w.lengths[:k], name=f"{w.name}; its first {k} request(s) only")
    if args.sweep is not None:
        if rank == 0:
            run_sweep(args, w)
        return
    if args.impl == "reference":
        line = run_reference(args, w, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    res = run_gb300(args, w, rank, world)
    if rank != 0:
        return
    pk, pk_kind = peaks()
    ms = res["ms"]
    T_all = w.T * world
    summ = summarize(w, res, pk, pk_kind)
    line = {"metric": METRIC, "value": T_all / (ms * 1e-3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": workload_config(w),
            "roofline": summ.pop("roofline"), "gpu_launches": int(res["launches"]), "clocks": res["clocks"],
            "score_select_compact_tokens_per_s": T_all / (summ["score_select_compact_ms"] * 1e-3),
            "kept_tokens": res["kept"], "kstar": res["kstar"][:8], "ms_per_step_spread": res["spread"],
            "eager_ms_per_step": res["eager_ms"], "launches_per_step": res["per_step_launches"],
            "near_threshold_blocks": res["near_threshold"], "stages": summ["stages"]}
    if not args.no_e2e:
        line["e2e"] = e2e_measure(args, w, res)
    if world == 1 and not args.no_cpu_baseline:
        sample = min(w.T, 32768)
        sw = oracle_sample(w, sample)
        sec = oracle_once(*sw)
        line["cpu_baseline"] = {"value": sample / sec, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                                "seconds": sec,
                                "sample": (f"the whole workload ({sample} tokens)" if sw[0] is w else
                                           f"one request of {sample} tokens with the workload's geometry")
                                          + ": score+select+compact+scatter in fp64 numpy, inputs excluded"}
    if world == 1 and not args.no_per_config:
        # the other workloads, each measured the same way (graph replays, L2 flushed, events on the stream)
        del res
        _free_device_memory()
        per = {}
        for i in sorted(recipe.CONFIGS):
            if i == args.config:
                continue
            wi = recipe.workload(i)
            ri = run_gb300(args, wi, rank, world, steps=max(3, args.per_config_steps), sample_clocks=False)
            si = summarize(wi, ri, pk, pk_kind)
            per[str(i)] = {"workload": wi.name, "R": wi.R, "T": wi.T, "Hq": wi.Hq, "Hkv": wi.Hkv, "d_k": wi.dk,
                           "hidden": wi.hdim, "G": wi.G, "n": wi.n, "p": wi.p,
                           "tokens_per_s": wi.T / (ri["ms"] * 1e-3), "ms_per_step": ri["ms"],
                           "score_select_compact_tokens_per_s": wi.T / (si["score_select_compact_ms"] * 1e-3),
                           "rho": ri["kept"] / max(1, wi.T), "kept_tokens": ri["kept"],
                           "kstar": {"min": int(min(ri["kstar"])), "max": int(max(ri["kstar"])),
                                     "first": [int(k) for k in ri["kstar"][:4]]},
                           "near_threshold_blocks": ri["near_threshold"],
                           "launches_per_step": ri["per_step_launches"], "steps": max(3, args.per_config_steps),
                           "roofline": si["roofline"], "stages": si["stages"]}
            del ri
            _free_device_memory()
        line["per_config"] = per
    print(json.dumps(line), flush=True)


def _free_device_memory():
    import gc
    import torch
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def summarize(w, res, pk, pk_kind):
    """Stage times and roofline fractions of one measured workload (eager breakdown of run_gb300)."""
    st = res["stage_ms"]
    names = ["score", "select", "compact", "slot_mapping", "scatter_back", "seqused"]
    kept = res["kept"]
    flops = score_flops(w)
    bytes_rows = 2 * kept * w.hdim * 2                           # read + write of every kept row
    stages = {nm: {"ms": float(st[i])} for i, nm in enumerate(names)}
    sbytes = score_input_bytes(w)
    stages["score"].update({"tflops": flops / (st[0] * 1e-3) / 1e12,
                            "frac_of_bf16_peak": flops / (st[0] * 1e-3) / 1e12 / pk["bf16_tflops"],
                            "input_gbs": sbytes / (st[0] * 1e-3) / 1e9,
                            "frac_of_hbm": sbytes / (st[0] * 1e-3) / 1e9 / pk["hbm_gbs"]})
    for nm in ("compact", "scatter_back"):
        i = names.index(nm)
        gbs = (bytes_rows + kept * 4) / (st[i] * 1e-3) / 1e9
        stages[nm].update({"gbs": gbs, "frac_of_hbm": gbs / pk["hbm_gbs"]})
    stages["select"]["us"] = float(st[1] * 1e3)
    # roofline of the dominant kernel: the row copy (up_scatter_back is exactly one launch of it, and the
    # same copy does compaction's gather); the score call is reported under "stages"
    sc_ms = float(st[4])
    row_bytes = bytes_rows + kept * 4
    rl = {"bound": "hbm", "kernel": "rows_kernel (up_scatter_back: one launch per step)",
          "achieved": row_bytes / (sc_ms * 1e-3) / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
          "algorithmic_bytes": row_bytes}
    rl["frac"] = rl["achieved"] / rl["peak"]
    rl["traffic"] = measured_traffic("rows_kernel", w)
    rl["peak_source"] = pk_kind
    return {"stages": stages, "roofline": rl, "score_select_compact_ms": float(st[0] + st[1] + st[2])}


if __name__ == "__main__":
    main()
