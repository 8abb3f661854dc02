"""Decode throughput of the persistent MoE megakernel on the full-scale synthetic model.

Workload (one GPU): the full-scale synthetic MoE shaped to the pages' model
(48 layers, d 2048, 32 query / 4 KV heads of 128, 128 experts top-8 with
F 768, vocab 152064, untied LM head; ~6.1 GB of active bf16 weights per
token) at batch 1 with 8192 cached tokens, greedy decoding.  A "step" is one
mk_decode_step: every layer's norm, QKV, RoPE + KV append, paged attention,
router top-k, expert SwiGLU, output projection and residual, then the final
norm, LM head and argmax -- one persistent kernel launch.

Metric: decode tokens/s and the fraction of the HBM speed of light, where
SOL time = algorithmic bytes (active weights from the observed routing + KV
read) / measured HBM bandwidth (MEASURED_PEAKS.json).  Inputs are larger
than L2 (6.9 GB streamed per step), so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mk|reference]

--impl reference times the CPU oracle (the plain reference of the same step)
on this machine's host cores, on a bounded sample of the same workload.
Under torchrun each rank runs an independent replica (the path does not
shard): weak scaling, max-over-ranks timing.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tok/s at batch 1/8 and % of HBM speed-of-light (bytes/step ÷ peak GB/s)"
PEAK_FALLBACK_GBS = 6800.0


HEADLINE_WORKLOAD = ("full-scale synthetic MoE, batch 1 at 8192 cached tokens (48 layers, d 2048, "
                     "32/4 heads x 128, 128 experts top-8, F 768, vocab 152064)")


def headline_config(lens, steps, world=1):
    """The config dict of the headline line (both arms print the same one)."""
    return {"workload": HEADLINE_WORKLOAD, "batch": len(lens), "cached_tokens": list(lens),
            "decode_steps": steps,
            "l2": "inputs larger than L2 (6.9 GB streamed per step), no flush",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return PEAK_FALLBACK_GBS, "fallback"


def weight_bytes_step(dims, sum_u_layers: float, batch: int) -> float:
    """Algorithmic weight bytes of one step: attention projections, router,
    norms, the distinct chosen experts (sum over layers of U_l), LM head,
    final norm and the embedding rows."""
    d, D, Hq, Hkv = dims.d_model, dims.head_dim, dims.n_q_heads, dims.n_kv_heads
    E, F, V, L = dims.n_experts, dims.d_ffn, dims.vocab, dims.n_layers
    per_layer = d * (Hq + 2 * Hkv) * D + Hq * D * d + E * d + d
    return 2.0 * (L * per_layer + sum_u_layers * 3 * d * F + V * d + d + batch * d)


def kv_bytes_step(dims, lens) -> float:
    """K and V bytes read for one step: L_b + 1 positions per sequence."""
    return float(sum(L + 1 for L in lens)) * dims.n_layers * 2 * dims.n_kv_heads * dims.head_dim * 2


def sol_formula(bytes_per_step: float, bw_gbs: float, batch: int = 1) -> float:
    """Speed-of-light tokens/s: batch tokens per (bytes / bandwidth)."""
    return batch * bw_gbs * 1e9 / bytes_per_step


def kernel_source_hash() -> str:
    """Hash of the kernel's compile inputs (its source and the headers that
    fix its limits and layouts)."""
    h = hashlib.sha256()
    for name in ("mk_kernel.cu", "mk_internal.h"):
        with open(os.path.join(ROOT, "persistent_moe_decode_sm_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "mk_decode_kernel_full_b1_8k.md")
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", txt)
    if not m or not h or h.group(1) != kernel_source_hash():
        return None
    return float(m.group(1))


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"mk_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        self.proc.wait()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------------ GPU arm


def run_mk(args, rank, world):
    import torch

    import persistent_moe_decode_sm_gb300 as mk
    import synth

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    wl = synth.workloads()["full"]
    dims = wl.dims
    if args.layers:
        # profiling captures only: the same model cut to its first layers
        dims = dataclasses.replace(dims, n_layers=args.layers)
    lens = list(wl.seq_lens) * args.batch
    B = len(lens)
    e2e_steps = args.e2e_steps
    reserve = args.warmup + args.steps + e2e_steps + 8
    inp = synth.device_inputs(dims, lens, reserve, None, seed=0)
    pl = inp.layout
    stream = torch.cuda.current_stream(dev)
    dec = mk.Decoder(dims, inp.tensors, pl.num_pages, pl.max_pages, max(B, 1),
                     inp.bias_tensors, stream)
    dec.build_schedule(lens, pl.page_tables)
    tok = [torch.tensor(synth.first_tokens(dims, B), dtype=torch.int32, device=dev),
           torch.zeros(B, dtype=torch.int32, device=dev)]
    logits = torch.empty(B, dims.vocab, dtype=torch.float32, device=dev)

    # warm-up (greedy: each step's argmax is the next step's input)
    cur = 0
    for _ in range(args.warmup):
        dec.decode_step(tok[cur], logits, tok[cur ^ 1])
        cur ^= 1
    dec.sync()
    st0 = dec.stats()
    lens_at_start = [L + args.warmup for L in lens]

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index)
    sampler.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(args.steps):
        ev[k][0].record(stream)
        dec.decode_step(tok[cur], logits, tok[cur ^ 1])
        ev[k][1].record(stream)
        cur ^= 1
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    dec.sync()
    total_ms = t_start.elapsed_time(t_end)
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    if world > 1:
        t = torch.tensor([total_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    st1 = dec.stats()
    sum_u = float(st1.sum_experts - st0.sum_experts)  # over steps and layers

    # algorithmic bytes over the timed steps
    w_bytes = sum(weight_bytes_step(dims, 0.0, B) for _ in range(args.steps)) + \
        2.0 * sum_u * 3 * dims.d_model * dims.d_ffn
    kv_bytes = sum(kv_bytes_step(dims, [L + k for L in lens_at_start]) for k in range(args.steps))
    total_bytes = w_bytes + kv_bytes
    bytes_per_step = total_bytes / args.steps
    peak, peak_kind = load_peaks()
    secs = total_ms / 1e3
    tok_s = B * args.steps / secs * world
    sol_tok_s = sol_formula(bytes_per_step, peak, B)
    mean_launch_s = statistics.mean(launch_ms) / 1e3
    achieved_gbs = bytes_per_step / mean_launch_s / 1e9

    # end to end through the C ABI with host buffers: H2D of the token ids,
    # the step, D2H of the next tokens, every step
    h_tok = torch.tensor(synth.first_tokens(dims, B), dtype=torch.int32).pin_memory()
    h_next = torch.empty(B, dtype=torch.int32).pin_memory()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        tok[0].copy_(h_tok, non_blocking=True)
        dec.decode_step(tok[0], logits, tok[1])
        h_next.copy_(tok[1], non_blocking=True)
        stream.synchronize()
        h_tok.copy_(h_next)
    e2e_s = time.perf_counter() - t0
    dec.sync()
    e2e_tok_s = B * e2e_steps / e2e_s * world if e2e_steps else None
    trace_summary = None
    if args.trace:
        # one more step with the per-task trace on (outside the timed region)
        from persistent_moe_decode_sm_gb300 import trace as mktrace

        mk.mk_set_trace(dec.ctx, dims.n_layers * 16 + 16)
        mk.mk_set_stage_trace_cta(dec.ctx, args.trace_cta)
        dec.decode_step(tok[0], logits, tok[1])
        tr, stages = mk.mk_get_trace(dec.ctx)
        trace_summary = mktrace.summarize(tr, dims.n_layers)
        trace_summary["stages_cta"] = args.trace_cta
        trace_summary["stages"] = mktrace.stage_summary(stages)
        if args.trace_raw:
            import numpy as np

            np.savez_compressed(args.trace_raw, tasks=tr, stages=stages)
        with open(args.trace, "w") as f:
            json.dump(trace_summary, f, indent=1)
        mk.mk_set_trace(dec.ctx, 0)
    dec.close()
    weights = {n: inp.tensors[n] for n in synth.weight_specs(dims)}
    del inp

    out = {
        "metric": METRIC, "value": round(tok_s, 2), "unit": "tok/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded bf16 N(0,0.02) weights, N(0,1) KV; no trained weights)",
        "config": (headline_config(lens, args.steps, world) if not args.layers and B == 1 else
                   {**headline_config(lens, args.steps, world),
                    "workload": f"profiling cut of the full-scale synthetic MoE: {dims.n_layers} layers, "
                                f"batch {B} at {lens[0]} cached tokens (not a bench line)"}),
        "sol": {"bytes_per_step": round(bytes_per_step), "weight_bytes_per_step":
                round(w_bytes / args.steps), "kv_bytes_per_step": round(kv_bytes / args.steps),
                "sol_tok_s": round(sol_tok_s, 1), "fraction": round(tok_s / world / sol_tok_s, 4),
                "bw_gbs": peak, "bw_kind": peak_kind},
        "roofline": {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved_gbs / peak, 4),
                     "traffic": profiled_traffic() if B == 1 else None,
                     "kernel": f"mk::decode_kernel<{1 if B <= 1 else 2 if B <= 2 else 4 if B <= 4 else 8}>",
                     "peak_kind": f"{peak_kind} (copy bandwidth)",
                     "mean_launch_ms": round(mean_launch_s * 1e3, 4)},
        "e2e": {"value": e2e_tok_s and round(e2e_tok_s, 2), "unit": "tok/s", "h2d_bytes_per_step": 4 * B,
                "d2h_bytes_per_step": 4 * B, "steps": e2e_steps},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if trace_summary:
        out["trace"] = {k: trace_summary[k] for k in ("step_us", "layer_us_median", "cta_time_split")}
    batches = [int(x) for x in args.batches.split(",") if x.strip()]
    if batches and world == 1 and not args.layers:
        out["batches"] = batch_sweep(dims, dev, stream, batches, weights)
    if args.workloads and world == 1 and not args.layers:
        out["workloads"] = other_workloads(dev, stream, weights, args.workloads.split(","))
    return out


def batch_sweep(dims, dev, stream, batches, weights, steps=64, warmup=4):
    """Decode tok/s and speed-of-light fraction of the same full-scale model
    at other batch sizes, every sequence at 8192 cached tokens (CUDA-event
    timed runs after the headline measurement)."""
    import torch

    import persistent_moe_decode_sm_gb300 as mk
    import synth

    if not batches:
        return []
    lens_all = [8192] * max(batches)
    inp = synth.device_inputs(dims, lens_all, warmup + steps + 8, None, seed=0, weights=weights)
    pl = inp.layout
    peak, _ = load_peaks()
    res = []
    for B in batches:
        lens = lens_all[:B]
        dec = mk.Decoder(dims, inp.tensors, pl.num_pages, pl.max_pages, B, inp.bias_tensors, stream)
        dec.build_schedule(lens, pl.page_tables[:B])
        tok = [torch.tensor(synth.first_tokens(dims, B), dtype=torch.int32, device=dev),
               torch.zeros(B, dtype=torch.int32, device=dev)]
        logits = torch.empty(B, dims.vocab, dtype=torch.float32, device=dev)
        cur = 0
        for _ in range(warmup):
            dec.decode_step(tok[cur], logits, tok[cur ^ 1])
            cur ^= 1
        dec.sync()
        st0 = dec.stats()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            dec.decode_step(tok[cur], logits, tok[cur ^ 1])
            cur ^= 1
        b.record(stream)
        torch.cuda.synchronize()
        dec.sync()
        ms = a.elapsed_time(b)
        sum_u = float(dec.stats().sum_experts - st0.sum_experts)
        w = steps * weight_bytes_step(dims, 0.0, B) + 2.0 * sum_u * 3 * dims.d_model * dims.d_ffn
        kv = sum(kv_bytes_step(dims, [L + warmup + k for L in lens]) for k in range(steps))
        per_step = (w + kv) / steps
        tok_s = B * steps / (ms / 1e3)
        sol = sol_formula(per_step, peak, B)
        res.append({"batch": B, "cached_tokens": 8192, "tok_s": round(tok_s, 2),
                    "ms_per_step": round(ms / steps, 4), "bytes_per_step": round(per_step),
                    "sol_tok_s": round(sol, 1), "sol_fraction": round(tok_s / sol, 4),
                    "steps": steps, "warmup": warmup})
        dec.close()
    del inp
    return res


def timed_decode(dec, dims, dev, stream, lens0, tokens0, steps, warmup, events=(), spare=None):
    """Greedy decode: `warmup` untimed steps, then `steps` steps between two
    CUDA events.  events: (step, slot) replacements inside the timed region
    (continuous batching): the slot takes the next spare sequence (length,
    page row, first token) and the schedule is rebuilt -- host work that the
    events' interval includes.  Returns (ms, sum of U over the timed steps,
    KV bytes read over the timed steps, replacements done)."""
    import numpy as np
    import torch

    B = len(lens0)
    lens = list(lens0)
    pt = np.array(spare["page_rows"][:B], copy=True) if spare else None
    tok = [torch.tensor(tokens0, dtype=torch.int32, device=dev),
           torch.zeros(B, dtype=torch.int32, device=dev)]
    logits = torch.empty(B, dims.vocab, dtype=torch.float32, device=dev)
    cur = 0
    for _ in range(warmup):
        dec.decode_step(tok[cur], logits, tok[cur ^ 1])
        cur ^= 1
        lens = [L + 1 for L in lens]
    dec.sync()
    st0 = dec.stats()
    ev = sorted(events)
    at, used, kv = 0, 0, 0.0
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for k in range(steps):
        changed = False
        while at < len(ev) and ev[at][0] == k:
            slot = ev[at][1]
            j = B + used
            lens[slot] = spare["lens"][j]
            pt[slot] = spare["page_rows"][j]
            tok[cur][slot] = int(spare["tokens"][used])
            used += 1
            at += 1
            changed = True
        if changed:
            dec.build_schedule(lens, pt)
        kv += kv_bytes_step(dims, lens)
        dec.decode_step(tok[cur], logits, tok[cur ^ 1])
        cur ^= 1
        lens = [L + 1 for L in lens]
    b.record(stream)
    torch.cuda.synchronize()
    dec.sync()
    return a.elapsed_time(b), float(dec.stats().sum_experts - st0.sum_experts), kv, used


def other_workloads(dev, stream, weights, names):
    """The other workloads, each on its own KV pool (the full-scale ones
    reuse the headline's weights):
      mid: the 8-layer mid model, batch 1 at 2048 cached tokens, 128 steps
           (its 225 MB partly fit L2, so its SOL fraction is informational);
      full_b8: batch 8, ragged U[1024, 16384] contexts, Zipf(1.1) router
           bias, 256 steps with continuous batching: each slot's sequence
           has a budget ~U[16, 128] steps, then the slot takes a fresh
           sequence (fresh context and KV pages) and the schedule is
           rebuilt inside the timed region;
      long_b1 / long_b2: 262144 cached tokens at batch 1, 131072 at batch 2,
           64 steps."""
    import numpy as np
    import torch

    import persistent_moe_decode_sm_gb300 as mk
    import synth

    peak, _ = load_peaks()
    wl = synth.workloads()
    res = {}
    for name in names:
        name = name.strip()
        if name not in wl or name in ("full", "tiny"):
            continue
        w = wl[name]
        dims = w.dims
        lens0 = list(w.seq_lens)
        B = len(lens0)
        steps = w.steps
        warmup = 4
        events, spare = (), None
        layout_lens = list(lens0)
        if name == "full_b8":
            events = synth.replacement_events(0, B, steps)
            spare_lens = synth.ragged_lens(0, len(events), 1024, 16384, gen=1)
            layout_lens = lens0 + spare_lens
        inp = synth.device_inputs(dims, layout_lens, warmup + steps + 8, w.zipf_s, seed=0,
                                  weights=weights if dims == synth.FULL else None)
        pl = inp.layout
        if events:
            spare = {"lens": layout_lens, "page_rows": pl.page_tables,
                     "tokens": synth.first_tokens(dims, len(events), gen=1)}
        dec = mk.Decoder(dims, inp.tensors, pl.num_pages, pl.max_pages, B, inp.bias_tensors,
                         stream)
        dec.build_schedule(lens0, pl.page_tables[:B])
        ms, sum_u, kv, n_rep = timed_decode(dec, dims, dev, stream, lens0,
                                            synth.first_tokens(dims, B), steps, warmup, events,
                                            spare)
        dec.close()
        del inp
        torch.cuda.empty_cache()
        wb = steps * weight_bytes_step(dims, 0.0, B) + 2.0 * sum_u * 3 * dims.d_model * dims.d_ffn
        per_step = (wb + kv) / steps
        tok_s = B * steps / (ms / 1e3)
        sol = sol_formula(per_step, peak, B)
        r = {"batch": B, "cached_tokens": lens0 if B <= 2 else "ragged U[1024, 16384]",
             "steps": steps, "warmup": warmup, "tok_s": round(tok_s, 2),
             "ms_per_step": round(ms / steps, 4), "bytes_per_step": round(per_step),
             "bytes_basis": "active weights from the observed routing + KV read",
             "sol_tok_s": round(sol, 1), "sol_fraction": round(tok_s / sol, 4)}
        if name == "mid":
            r["sol_informational"] = "225 MB per step, partly L2-resident"
        if events:
            r["replacements"] = n_rep
            r["router_bias"] = "Zipf(1.1) per expert"
            r["schedule_rebuilds_in_timed_region"] = True
        res[name] = r
    return res


# -------------------------------------------------------------- CPU oracle


def oracle_step_time(max_seconds: float, max_steps: int, warmup: int = 0):
    """Times full-scale oracle decode steps (weights regenerated on the fly
    from the seeded generator) until max_steps or max_seconds, after
    `warmup` untimed steps."""
    import oracle
    import synth

    wl = synth.workloads()["full"]
    dims = wl.dims
    pl = synth.page_layout(dims, wl.seq_lens, max_steps + warmup + 2)
    host = synth.host_inputs(dims, pl, materialise=False)
    orc = oracle.Oracle(dims, host, wl.seq_lens, pl.page_tables)
    tok = synth.first_tokens(dims, 1)
    for _ in range(warmup):
        tok = orc.step(tok)["next_tokens"]
    times = []
    t_all = time.perf_counter()
    for _ in range(max_steps):
        t0 = time.perf_counter()
        r = orc.step(tok)
        times.append(time.perf_counter() - t0)
        tok = r["next_tokens"]
        if time.perf_counter() - t_all > max_seconds:
            break
    return times


def cpu_baseline(max_seconds=30.0, max_steps=3):
    times = oracle_step_time(max_seconds, max_steps)
    return {"value": round(len(times) / sum(times), 4), "unit": "tok/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{len(times)} full-scale decode step(s) of the oracle (batch 1, 8192 "
                      "cached tokens; weights regenerated on the fly from the seeded "
                      "generator, OpenMP over all host cores)"}


def run_reference(args):
    times = oracle_step_time(max_seconds=150.0, max_steps=max(1, args.steps), warmup=args.warmup)
    v = len(times) / sum(times)
    cb = {"value": round(v, 4), "unit": "tok/s", "cores": os.cpu_count(), "kind": "oracle",
          "sample": f"{len(times)} of the requested {args.steps} full-scale decode steps after "
                    f"{args.warmup} untimed ones (timed part bounded to ~150 s of CPU time); "
                    "weights regenerated on the fly"}
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "tok/s",
            "n_gpus": 1, "steps": len(times), "warmup": args.warmup,
            "ms_per_step": round(1e3 * sum(times) / len(times), 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32-accumulate over bf16",
            "data": "synthetic",
            "config": headline_config([8192], max(1, args.steps)),
            "cpu_baseline": cb,
            "e2e": {"value": round(v, 4), "unit": "tok/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="mk", choices=["mk", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batches", default="2,4,8",
                    help="also time these batch sizes at 8192 cached tokens ('' to skip)")
    ap.add_argument("--trace", default="", help="write a per-task trace summary (JSON) here")
    ap.add_argument("--trace-cta", type=int, default=0,
                    help="the CTA whose ring stages the trace records")
    ap.add_argument("--trace-raw", default="", help="also save the raw trace (npz) here")
    ap.add_argument("--workloads", default="mid,full_b8,long_b1,long_b2",
                    help="also time these workloads ('' to skip)")
    ap.add_argument("--batch", type=int, default=1,
                    help="profiling only: the headline step at this batch (8192 cached each)")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: cut the model to its first N layers")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    out = run_mk(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline()
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
