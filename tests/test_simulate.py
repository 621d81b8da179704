"""Pins for the cut predictor (Algorithm 1, SIMULATE, of "One Megakernel is
Not Enough: Predicting Where to Cut for Streaming Inference") on hand-worked
event graphs, and for the frame's cut compositions (Observation 3 of the same
paper: serial cuts under a fixed contract only add their dispatch cost)."""
import numpy as np
import pytest

from persistent_megakernel_streaming_gb300 import simulate as sim


def _two_launches(cta_each):
    """Launch 1 runs a (3) then b (2) one at a time, then its release r1
    (0.5); launch 2 runs c (4) then its release r2 (0). 132 CTAs."""
    nodes = ["a", "b", "r1", "c", "r2"]
    preds = {"b": ["a"], "r1": ["a", "b"], "r2": ["c"]}
    T = {"a": 3.0, "b": 2.0, "r1": 0.5, "c": 4.0, "r2": 0.0}
    launch = {"a": 1, "b": 1, "c": 2}
    cta = {1: cta_each, 2: cta_each}
    return nodes, preds, T, launch, cta, {1: 1, 2: 1}, {1: "r1", 2: "r2"}


def test_two_launches_that_cannot_share_the_gpu_run_one_after_the_other():
    """100 + 100 CTAs > 132: launch 2 is admitted only when r1 frees launch
    1's CTAs at 3 + 2 + 0.5 = 5.5, so c runs 5.5 .. 9.5."""
    nodes, preds, T, launch, cta, mt, rel = _two_launches(100)
    fin = sim.simulate(nodes, preds, T, launch, cta, mt, rel, ncta=132)
    assert fin == {"a": 3.0, "b": 5.0, "r1": 5.5, "c": 9.5, "r2": 9.5}


def test_two_launches_that_fit_together_overlap():
    """60 + 60 CTAs fit: both are admitted at 0, c runs 0 .. 4 beside a and b."""
    nodes, preds, T, launch, cta, mt, rel = _two_launches(60)
    fin = sim.simulate(nodes, preds, T, launch, cta, mt, rel, ncta=132)
    assert fin == {"a": 3.0, "b": 5.0, "r1": 5.5, "c": 4.0, "r2": 4.0}


def test_max_tasks_serialises_a_launch():
    """Three independent unit tasks of one launch, at most two at a time:
    two finish at 1, the third at 2."""
    nodes = ["x", "y", "z", "r"]
    preds = {"r": ["x", "y", "z"]}
    T = {"x": 1.0, "y": 1.0, "z": 1.0, "r": 0.0}
    fin = sim.simulate(nodes, preds, T, {"x": 0, "y": 0, "z": 0}, {0: 10}, {0: 2}, {0: "r"}, ncta=10)
    assert (fin["x"], fin["y"], fin["z"], fin["r"]) == (1.0, 1.0, 2.0, 2.0)


def test_memory_demand_shares_the_bandwidth():
    """Two unit tasks each demanding the whole bandwidth run at half speed and
    finish at 2; half the bandwidth each, they run at full speed. A task
    alone demanding twice the bandwidth runs at half speed (2), beside a task
    with no demand (3)."""
    nodes = ["p", "q"]
    fin = sim.simulate(nodes, {}, {"p": 1.0, "q": 1.0}, Q={"p": 1.0, "q": 1.0}, bmem=1.0)
    assert fin == {"p": 2.0, "q": 2.0}
    fin = sim.simulate(nodes, {}, {"p": 1.0, "q": 1.0}, Q={"p": 0.5, "q": 0.5}, bmem=1.0)
    assert fin == {"p": 1.0, "q": 1.0}
    fin = sim.simulate(nodes, {}, {"p": 1.0, "q": 3.0}, Q={"p": 2.0}, bmem=1.0)
    assert fin == {"p": 2.0, "q": 3.0}


def test_deadlock_is_reported():
    """A launch that holds more CTAs than the device has never starts."""
    with pytest.raises(sim.Deadlock):
        sim.simulate(["a", "r"], {"r": ["a"]}, {"a": 1.0, "r": 0.0}, {"a": 0}, {0: 200}, {0: 1}, {0: "r"},
                     ncta=132)
    with pytest.raises(sim.Deadlock):  # a cycle: nothing is ever ready
        sim.simulate(["a", "b"], {"a": ["b"], "b": ["a"]}, {"a": 1.0, "b": 1.0})


def test_serial_cuts_add_only_their_dispatch_cost():
    """The frame as k+1 consecutive full-grid launches: with no dispatch cost
    the simulated frame equals the single launch (Observation 3); with a cost
    d per launch it grows by exactly k * d."""
    rng = np.random.default_rng(3)
    ph = list(rng.uniform(1.0, 9.0, size=432))
    single = sim.predict_frame_us(ph, [], 0.0)
    assert abs(single - sum(ph)) < 1e-9
    for cuts in ([216], [2 + 27 * i for i in range(1, 16)], sorted(rng.choice(np.arange(1, 432), 80, False))):
        assert abs(sim.predict_frame_us(ph, cuts, 0.0) - single) < 1e-9
        assert abs(sim.predict_frame_us(ph, cuts, 6.5) - (single + 6.5 * len(cuts))) < 1e-9


def test_calibration_recovers_the_dispatch_cost():
    rng = np.random.default_rng(4)
    ph = list(rng.uniform(1.0, 9.0, size=100))
    frame = sum(ph) * 1.01
    d, scaled = sim.calibrate_dispatch(ph, 50, frame + 7.25, frame)
    assert abs(d - 7.25) < 1e-9 and abs(sum(scaled) - frame) < 1e-9
    assert abs(sim.predict_frame_us(scaled, [10, 50, 90], d) - (frame + 3 * 7.25)) < 1e-9
    d, _ = sim.calibrate_dispatch(ph, [20, 40, 60, 80], frame + 4 * 6.5, frame)
    assert abs(d - 6.5) < 1e-9


def test_bad_cuts_are_refused():
    with pytest.raises(ValueError):
        sim.frame_event_graph([1.0] * 10, [5, 5], 1.0)
    with pytest.raises(ValueError):
        sim.frame_event_graph([1.0] * 10, [10], 1.0)
