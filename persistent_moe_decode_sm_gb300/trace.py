"""Summaries of the kernel's per-task trace (mk_set_trace / mk_get_trace).

Each event is one task run by one CTA: entry, dependency satisfied, first
data stage available, exit (globaltimer ns).  `summarize` reports, per
phase (op) averaged over layers, when the phase starts and ends relative to
the previous layer's end, and, over all CTAs, how the time splits into
waiting for a dependency, waiting for data, and working.
"""
from __future__ import annotations

from collections import defaultdict

import numpy as np

OPS = {1: "qkv", 2: "router", 3: "attn", 4: "up", 5: "out", 6: "lm", 7: "down"}


def events(trace: np.ndarray):
    """Flat list of (cta, op, layer, task, t_entry, t_ready, t_stage, t_exit,
    stage_wait_ns, n_stages, t_mark)."""
    out = []
    for c in range(trace.shape[0]):
        for e in trace[c]:
            if e[1] == 0:
                continue
            w = int(e[0])
            out.append((c, w & 0xFF, (w >> 8) & 0xFFF, w >> 20, int(e[1]), int(e[2]), int(e[3]),
                        int(e[4]), int(e[5]), int(e[6]), int(e[7])))
    return out


def summarize(trace: np.ndarray, n_layers: int) -> dict:
    ev = events(trace)
    if not ev:
        return {}
    t0 = min(e[4] for e in ev)
    t_end = max(e[7] for e in ev)
    per = defaultdict(list)
    for e in ev:
        per[(e[2], e[1])].append(e)
    layer_end = {}
    for l in range(n_layers):
        ends = [e[7] for k, v in per.items() if k[0] == l for e in v]
        if ends:
            layer_end[l] = max(ends)
    phase = defaultdict(lambda: defaultdict(list))
    for (l, op), v in per.items():
        if op == 6 or l == 0 or l not in layer_end or (l - 1) not in layer_end:
            continue
        base = layer_end[l - 1]
        phase[OPS[op]]["p50_ready_us"].append((float(np.median([e[5] for e in v])) - base) / 1e3)
        phase[OPS[op]]["p50_exit_us"].append((float(np.median([e[7] for e in v])) - base) / 1e3)
        phase[OPS[op]]["first_entry_us"].append((min(e[4] for e in v) - base) / 1e3)
        phase[OPS[op]]["last_ready_us"].append((max(e[5] for e in v) - base) / 1e3)
        st = [e[6] for e in v if e[6]]
        if st:
            phase[OPS[op]]["last_first_stage_us"].append((max(st) - base) / 1e3)
        phase[OPS[op]]["last_exit_us"].append((max(e[7] for e in v) - base) / 1e3)
        phase[OPS[op]]["mean_busy_us"].append(np.mean([(e[7] - max(e[5], e[6] or e[5])) / 1e3
                                                       for e in v]))
        phase[OPS[op]]["mean_stage_wait_us"].append(np.mean([e[8] / 1e3 for e in v]))
        phase[OPS[op]]["mean_stages"].append(np.mean([e[9] for e in v]))
        mk = [(e[10] - max(e[5], e[6] or e[5])) / 1e3 for e in v if e[10]]
        if mk:
            phase[OPS[op]]["mean_to_mark_us"].append(np.mean(mk))
    phases = {op: {k: round(float(np.median(v)), 2) for k, v in d.items()}
              for op, d in phase.items()}
    layer_times = [(layer_end[l] - layer_end[l - 1]) / 1e3 for l in range(1, n_layers)
                   if l in layer_end and l - 1 in layer_end]
    wait_dep = sum(e[5] - e[4] for e in ev)
    wait_data = sum(max(0, e[6] - e[5]) for e in ev if e[6])
    busy = sum(e[7] - max(e[5], e[6] or e[5]) for e in ev)
    total = (t_end - t0) * trace.shape[0]
    return {
        "step_us": round((t_end - t0) / 1e3, 1),
        "layer_us_median": round(float(np.median(layer_times)), 2) if layer_times else None,
        "lm_head_us": round((t_end - layer_end.get(n_layers - 1, t0)) / 1e3, 2),
        "cta_time_split": {"wait_dependency": round(wait_dep / total, 3),
                           "wait_first_data": round(wait_data / total, 3),
                           "task_body": round(busy / total, 3)},
        "phases_rel_prev_layer_end_us": phases,
    }


def stage_times_ns(stages: np.ndarray) -> np.ndarray:
    """The stage events with their SM-clock columns converted to globaltimer
    nanoseconds (through the anchor pair in the last event)."""
    a = stages[-1].astype(np.float64)
    out = stages[:-1].astype(np.float64).copy()
    if a[3] <= a[1]:
        return out
    ns_per_clk = (a[2] - a[0]) / (a[3] - a[1])
    for c in range(1, 8):
        nz = out[:, c] != 0
        out[nz, c] = a[0] + (out[nz, c] - a[1]) * ns_per_clk
    return out


def stage_summary(stages: np.ndarray) -> dict:
    """Per op, medians over CTA 0's ring stages (microseconds): the producer's
    time to find the next stage (desc), to get its slot back (slot_wait),
    to issue the copies (issue); the copy latency (issue -> data seen by the
    owning warp, counting from when the warp started waiting if later); the
    owning warp's wait and compute (data seen -> release); and the stage
    interval (producer issue to issue)."""
    ev = [e for e in stage_times_ns(stages) if e[4] and e[6] and e[7]]
    if not ev:
        return {}
    out = {}
    issue = np.array(sorted(int(e[4]) for e in ev), np.int64)
    per = defaultdict(list)
    for e in ev:
        per[OPS.get((int(e[0]) >> 24) & 0xFF, "?")].append(e)
    for op, v in per.items():
        a = np.array([[int(x) for x in e] for e in v], np.int64)
        out[op] = {
            "n": len(v),
            "desc_us": round(float(np.median(a[:, 2] - a[:, 1])) / 1e3, 3),
            "slot_wait_us": round(float(np.median(a[:, 3] - a[:, 2])) / 1e3, 3),
            "issue_us": round(float(np.median(a[:, 4] - a[:, 3])) / 1e3, 3),
            "copy_latency_us": round(float(np.median(a[:, 6] - a[:, 4])) / 1e3, 3),
            "warp_wait_us": round(float(np.median(a[:, 6] - a[:, 5])) / 1e3, 3),
            "compute_us": round(float(np.median(a[:, 7] - a[:, 6])) / 1e3, 3),
        }
    out["issue_interval_us"] = round(float(np.median(np.diff(issue))) / 1e3, 3) if len(issue) > 1 else None
    return out
