"""Where to cut the frame into launches: the event-graph simulation of
"One Megakernel is Not Enough: Predicting Where to Cut for Streaming
Inference" (Algorithm 1, SIMULATE), and its event graph for this frame.

Host-side planning tool; nothing here runs on the GPU or on the frame's path.

SIMULATE (section "Megakernel Impact Simulation", Algorithm 1) advances an
event graph in time. Every node has a standalone service time and may belong
to a launch; a launch holds its CTAs from admission until its release node
completes, admits only while enough CTAs are free, and runs at most
`max_tasks` of its nodes at once. Running nodes with a memory demand share
the device bandwidth: each progresses at min(1, B / total demand). A ready
node that can never be admitted leaves nothing running: a deadlock.

The frame's event graph (section "Event Graph (evGraph)" and Table I's
"Event graph" rows): each phase is one node whose service time is the span it
takes inside the single persistent launch (measured with cp_trace), the
phases of a frame form a chain, and a cut composition splits the chain into
consecutive launches that each hold every CTA of the grid. A launch is a
dispatch node (the per-launch cost: a launch can only start once the previous
one has released its CTAs, then runs its prologue and streams its first
weights cold), its phases, and a release node. Observation 3 of the same
paper is what this predicts for serial cuts under a fixed contract: the
device schedule is unchanged and each cut adds its dispatch cost.
"""
from __future__ import annotations

from collections import deque


class Deadlock(RuntimeError):
    """Nodes remain but none can run (SIMULATE's DEADLOCK)."""


def simulate(nodes, preds, T, launch=None, cta=None, max_tasks=None, release=None, Q=None,
             bmem=None, ncta=0):
    """Algorithm 1 of "One Megakernel is Not Enough", section "Megakernel
    Impact Simulation".

    nodes: node ids in a fixed order (READY is scanned in the order nodes
      become ready, ties in this order).
    preds: {v: [predecessors]} (missing: none).
    T: {v: standalone service time}.
    launch: {v: launch id or None}; cta: {L: CTAs L holds}; max_tasks:
      {L: nodes of L that may run at once}; release: {L: node whose
      completion frees L's CTAs}.
    Q: {v: memory demand, bytes per unit time while running} (missing: 0);
      bmem: device memory bandwidth in the same units; ncta: CTAs of the device.

    Returns {v: finish time}; raises Deadlock when nodes remain and none runs.
    """
    launch = launch or {}
    cta = cta or {}
    max_tasks = max_tasks or {}
    release = release or {}
    Q = Q or {}
    succ = {v: [] for v in nodes}
    npred = {v: 0 for v in nodes}
    for v in nodes:
        for u in preds.get(v, ()):
            succ[u].append(v)
            npred[v] += 1
    rel_of = {r: L for L, r in release.items()}
    t = 0.0
    rem = {v: float(T[v]) for v in nodes}
    left = dict(npred)
    ready = deque(v for v in nodes if npred[v] == 0)
    running, done, admitted = [], set(), set()
    free = ncta
    finish = {}
    while len(done) < len(nodes):
        # admit launches and start nodes, in READY order
        for v in list(ready):
            L = launch.get(v)
            if L is not None and L not in admitted and free >= cta[L]:
                admitted.add(L)
                free -= cta[L]
            if L is None or (L in admitted and sum(1 for u in running if launch.get(u) == L) < max_tasks[L]):
                ready.remove(v)
                running.append(v)
        if not running:
            raise Deadlock(f"{len(nodes) - len(done)} nodes left, none can run at t={t}")
        qtot = sum(Q.get(v, 0.0) for v in running)
        rate = {v: (1.0 if Q.get(v, 0.0) == 0 else min(1.0, bmem / qtot)) for v in running}
        dt = min(rem[v] / rate[v] for v in running)
        t += dt
        for v in running:
            rem[v] -= rate[v] * dt
        fin = [v for v in running if rem[v] <= 1e-12 * max(1.0, float(T[v]))]
        for v in fin:
            running.remove(v)
            finish[v] = t
            done.add(v)
            L = rel_of.get(v)
            if L is not None and L in admitted:
                admitted.discard(L)
                free += cta[L]
            for w in succ[v]:
                left[w] -= 1
                if left[w] == 0:
                    ready.append(w)
    return finish


def frame_event_graph(phase_us, cuts, dispatch_us, release_us=0.0, grid=144, phase_bytes=None, bmem=None):
    """The frame as len(cuts)+1 consecutive persistent launches.

    phase_us: service time of every phase, in frame order (the phase's span
      inside the single persistent launch).
    cuts: ascending phase indices, each starting a new launch.
    dispatch_us: per-launch cost paid before a launch's first phase (start
      after the previous launch's release, prologue, cold first weights);
      the first launch pays it too, so only differences between
      compositions are meaningful. release_us: the cost of a release node.
    phase_bytes (optional): weight bytes each phase streams; with bmem their
      demand (bytes / service time) shares the device bandwidth.

    Returns (nodes, preds, T, launch, cta, max_tasks, release, Q) for
    simulate() with ncta = grid, and the id of the last release node.
    """
    n = len(phase_us)
    bounds = [0] + [int(c) for c in cuts] + [n]
    if any(b <= a for a, b in zip(bounds, bounds[1:])):
        raise ValueError("cuts must be ascending phase indices inside the frame")
    nodes, preds, T, launch, Q = [], {}, {}, {}, {}
    cta, max_tasks, release = {}, {}, {}
    prev_release, prev_phase = None, None
    for i, (a, b) in enumerate(zip(bounds, bounds[1:])):
        d, r = ("dispatch", i), ("release", i)
        nodes.append(d)
        T[d] = float(dispatch_us)
        launch[d] = i
        preds[d] = [prev_release] if prev_release is not None else []
        cta[i], max_tasks[i], release[i] = grid, grid, r
        for k in range(a, b):
            v = ("phase", k)
            nodes.append(v)
            T[v] = float(phase_us[k])
            launch[v] = i
            preds[v] = [d] + ([prev_phase] if prev_phase is not None else [])
            if phase_bytes is not None and bmem:
                Q[v] = float(phase_bytes[k]) / max(float(phase_us[k]), 1e-12)
            prev_phase = v
        nodes.append(r)
        T[r] = float(release_us)
        launch[r] = None
        preds[r] = [("phase", b - 1)]
        prev_release = r
    return (nodes, preds, T, launch, cta, max_tasks, release, Q), prev_release


def predict_frame_us(phase_us, cuts, dispatch_us, release_us=0.0, grid=144, phase_bytes=None, bmem=None):
    """Simulated frame time of a cut composition: the finish of its last
    release node, less the first launch's dispatch (the single persistent
    launch, measured, includes its own start)."""
    g, last = frame_event_graph(phase_us, cuts, dispatch_us, release_us, grid, phase_bytes, bmem)
    nodes, preds, T, launch, cta, max_tasks, release, Q = g
    fin = simulate(nodes, preds, T, launch, cta, max_tasks, release, Q, bmem, grid)
    return fin[last] - float(dispatch_us)


def calibrate_dispatch(phase_us, cuts, measured_cut_us, measured_frame_us, release_us=0.0):
    """The per-launch cost that makes the simulated composition cut at `cuts`
    reproduce its measurement, with the phase service times scaled to
    reproduce the single launch (the paper's calibration of service times to
    standalone runs). Returns (dispatch_us, scaled phase_us)."""
    cuts = [cuts] if isinstance(cuts, int) else list(cuts)
    s = float(measured_frame_us) / float(sum(phase_us))
    scaled = [p * s for p in phase_us]
    # with dispatch d the composition simulates to (its value at d = 0) + len(cuts) * d
    base = predict_frame_us(scaled, cuts, 0.0, release_us)
    return (float(measured_cut_us) - base) / len(cuts), scaled
