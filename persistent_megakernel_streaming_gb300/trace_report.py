"""Per-task timestamp breakdown of one frame, from cp_trace output.

cp_trace gives, for every task of the static schedule, 16 int64 words of
%globaltimer nanoseconds (word 7 packs phase, kind and CTA):

  compute warps  0 task start, 1 dependencies satisfied (a projection with
                 per-chunk waits: its first input chunk's producers seen done),
                 2 inputs staged,
                 3 accumulator ready, 4 partial sums exchanged,
                 5 outputs stored, 6 signal issued
  MMA warp       8 accumulator free, 9 last weight page seen landed,
                 10 last input chunk ready, 12 MMAs committed
  producer warp  11 last weight page issued

The report splits each task into the steps the frame's critical path is made
of: wait (start -> dependencies), handoff (the predecessor phase's last
signal -> this task's dependencies seen), input landing (bulk copies of the
activations), the last weight page as the MMA warp first sees it, relative
to the dependency (it sees pages in order, so this is an upper bound on when
the page landed; negative: landed before the dependency), MMA (inputs staged
-> accumulator ready), exchange (K-split partials through distributed shared
memory), epilogue and signal. Per phase
kind it reports medians over tasks, and the sum over phases of each phase's
span (its last signal minus the previous phase's last signal), which adds up
to the frame.
"""
from __future__ import annotations

import numpy as np

KINDS = {0: "inproj", 1: "emb0", 2: "qkv", 3: "attn", 4: "o", 5: "gate_up", 6: "down", 7: "head", 8: "draw"}
PROJ = (0, 2, 4, 5, 6, 7)


def _med(x):
    x = x[np.isfinite(x)]
    return float(np.median(x)) if x.size else None


def breakdown(trace: np.ndarray) -> dict:
    """trace: int64 [tasks][16] from cp_trace. Returns a dict of per-kind
    step medians (microseconds) and per-kind totals of phase spans."""
    t = np.asarray(trace, dtype=np.int64)
    phase = t[:, 7] >> 32
    kind = (t[:, 7] >> 16) & 0xFFFF
    nph = int(phase.max()) + 1
    us = lambda a: a.astype(np.float64) / 1e3  # noqa: E731
    end = np.full(nph, -1, np.int64)
    for ph in range(nph):
        m = phase == ph
        if m.any():
            end[ph] = t[m, 6].max()
    t0 = t[t[:, 0] > 0, 0].min()
    frame_us = float(us(end.max() - t0))
    prev_end = np.zeros(len(t), np.int64)
    for ph in range(1, nph):
        prev_end[phase == ph] = end[ph - 1]
    span = {}
    for ph in range(nph):
        m = phase == ph
        if not m.any():
            continue
        k = KINDS.get(int(kind[m][0]), str(int(kind[m][0])))
        span[k] = span.get(k, 0.0) + float(us(end[ph] - (end[ph - 1] if ph > 0 else t0)))
    steps = {}
    for kk, name in KINDS.items():
        m = kind == kk
        if not m.any():
            continue
        T = t[m]
        has_prev = phase[m] > 0
        row = {"tasks": int(m.sum()),
               "wait": _med(us(T[:, 1] - T[:, 0])),
               "handoff": _med(us(T[has_prev, 1] - prev_end[m][has_prev])),
               "signal": _med(us(T[:, 6] - T[:, 5]))}
        if kk in PROJ:
            row.update({"inputs_land": _med(us(T[:, 2] - T[:, 1])),
                        "weights_seen_vs_dep": _med(us(T[:, 9] - T[:, 1])),
                        "mma": _med(us(T[:, 3] - T[:, 2])),
                        "exchange": _med(us(T[:, 4] - T[:, 3])),
                        "epilogue": _med(us(T[:, 5] - T[:, 4]))})
        else:
            row["body"] = _med(us(T[:, 5] - T[:, 1]))
        steps[name] = {k: (round(v, 3) if isinstance(v, float) else v) for k, v in row.items()}
    return {"frame_us": round(frame_us, 1), "phase_span_us_by_kind": {k: round(v, 1) for k, v in span.items()},
            "median_step_us_by_kind": steps}


def mma_stage_split(trace: np.ndarray) -> dict:
    """The projections' "mma" stage (inputs issued -> accumulator seen) split
    with the MMA warp's own stamps, medians in microseconds per kind:
    `land` inputs issued -> the last input chunk found landed by the MMA warp
    (which has issued the earlier chunks' MMAs by then), `tail` -> the last
    MMAs issued and committed, `complete` -> the compute warps see the
    accumulator (the MMAs finishing, the commit's barrier, the waiters
    waking)."""
    t = np.asarray(trace, dtype=np.int64)
    kind = (t[:, 7] >> 16) & 0xFFFF
    out = {}
    for kk in PROJ:
        m = (kind == kk) & (t[:, 2] > 0) & (t[:, 10] > 0) & (t[:, 12] > 0) & (t[:, 3] > 0)
        if not m.any():
            continue
        T = t[m]  # differences in integer nanoseconds first: the stamps are ~1e18
        d = lambda a, b: round(float(np.median((T[:, a] - T[:, b]).astype(np.float64))) / 1e3, 3)  # noqa: E731
        out[KINDS[kk]] = {"land": d(10, 2), "tail": d(12, 10), "complete": d(3, 12)}
    return out


def phase_spans(trace: np.ndarray) -> list:
    """Every phase's span in frame order, microseconds: its last signal minus
    the previous phase's last signal (the first phase from the earliest task
    start). They add up to the traced frame."""
    t = np.asarray(trace, dtype=np.int64)
    phase = t[:, 7] >> 32
    nph = int(phase.max()) + 1
    end = np.array([t[phase == ph, 6].max() for ph in range(nph)], dtype=np.int64)
    t0 = t[t[:, 0] > 0, 0].min()
    prev = np.concatenate([[t0], end[:-1]])
    return [float(x) / 1e3 for x in (end - prev)]


def tensor_utilisation(trace: np.ndarray, flops_by_kind: dict, peak_tflops: float) -> dict:
    """Per projection kind: its algorithmic flops over the frame (2 x weights
    x rows per phase) divided by the summed spans of its phases, as a
    fraction of the tensor peak. A phase's span is the time the frame spends
    on it, so this is the tensor pipe's share while that kind runs."""
    t = np.asarray(trace, dtype=np.int64)
    phase = t[:, 7] >> 32
    kind = (t[:, 7] >> 16) & 0xFFFF
    spans = phase_spans(t)
    out = {}
    for kk, name in KINDS.items():
        if name not in flops_by_kind:
            continue
        phs = sorted(set(int(x) for x in phase[kind == kk]))
        if not phs:
            continue
        us = sum(spans[ph] for ph in phs)
        tf = flops_by_kind[name] * len(phs) / (us * 1e-6) / 1e12
        out[name] = {"phases": len(phs), "tflops": round(tf, 2), "frac_of_peak": round(tf / peak_tflops, 4)}
    return out


def format_table(b: dict) -> str:
    """Plain-text table of a breakdown()."""
    cols = ["tasks", "handoff", "wait", "inputs_land", "weights_seen_vs_dep", "mma", "exchange", "epilogue",
            "body", "signal"]
    lines = [f"frame {b['frame_us']} us; phase spans by kind (us): {b['phase_span_us_by_kind']}",
             "median per task (us): " + " | ".join(cols)]
    for name, row in b["median_step_us_by_kind"].items():
        vals = []
        for c in cols:
            v = row.get(c)
            vals.append("-" if v is None else (str(v) if c == "tasks" else f"{v:.2f}"))
        lines.append(f"  {name:8s} " + " | ".join(vals))
    return "\n".join(lines)
