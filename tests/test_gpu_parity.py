"""GPU parity: the CUDA path through the C ABI against the oracle.

Element-by-element comparisons on seeded inputs, at sizes the oracle runs in
seconds (the tiny decoder; one to 64 rows of the full decoder), plus the
invariants that hold at any size: run-to-run bit identity, the persistent
frame equal to the per-phase graph, rows independent of the batch.
"""
import numpy as np
import pytest
import torch

import helpers
import oracle
from oracle import philox
from persistent_megakernel_streaming_gb300 import cp, torch_io

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


# ---------------------------------------------------------------- Philox
def test_philox_matches_oracle_and_curand():
    helpers.build.build()
    rng = np.random.default_rng(5)
    n = 4096
    ctr = rng.integers(0, 2 ** 32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    key = rng.integers(0, 2 ** 32, size=(n, 2), dtype=np.uint64).astype(np.uint32)
    ctr[:4] = 0
    key[:2] = 0xFFFFFFFF
    want = np.stack(philox.philox4x32(tuple(ctr.T.astype(np.uint64)), tuple(key.T.astype(np.uint64))), axis=1)
    tc = torch.from_numpy(ctr.view(np.int32)).cuda()
    tk = torch.from_numpy(key.view(np.int32)).cuda()
    for use_curand in (0, 1):
        out = torch.zeros((n, 4), dtype=torch.int32, device="cuda")
        cp.test_philox(tc, tk, use_curand, out)
        np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), want)


# ---------------------------------------------------------------- draw
def _draw_case(V, rows, seed):
    rng = np.random.default_rng(seed)
    lg = (rng.standard_normal((rows, V)) * 0.6).astype(np.float32)
    # plant exact ties in some rows (first and k-th place)
    lg[1, [3, 77]] = lg[1].max() + 0.5
    lg[2, :] = np.round(lg[2] * 4) / 4
    samp = dict(
        temperature=rng.choice([0.0, 0.3, 0.9, 1.2], size=rows).astype(np.float32),
        top_k=rng.choice([0, 1, 5, 20, 50, 200, V - 1, V], size=rows).astype(np.int32),
        top_p=rng.choice([1.0, 0.95, 0.8, 0.5, 0.1, 1e-6], size=rows).astype(np.float32),
        seed=rng.integers(0, 2 ** 63, size=rows, dtype=np.int64).astype(np.uint64),
        offset=rng.integers(0, 2 ** 40, size=rows, dtype=np.int64))
    samp["temperature"][:3] = 0.8
    return lg, samp


@pytest.mark.parametrize("V", [256, 2048])
def test_draw_matches_oracle(V):
    rows, group = 300, 3
    lg, samp = _draw_case(V, rows, 7 + V)
    codes = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
    cp.test_draw(torch.from_numpy(lg).cuda(), torch_io.sampler_to_torch(samp), group, codes)
    got = codes.cpu().numpy()
    mism = 0
    for r in range(rows):
        d = oracle.draw_detail(lg[r], samp["temperature"][r], samp["top_k"][r], samp["top_p"][r],
                               int(samp["seed"][r]), r, int(samp["offset"][r]) + group)
        if d["code"] != got[r]:
            # the two sides share the exact logits; only libm ulps can separate them
            assert d["margin"] < 1e-4 or d["topp_gap"] < 1e-5, (r, got[r], d)
            mism += 1
    assert mism <= 2


@pytest.mark.parametrize("step", [0.25, 0.125])
def test_draw_with_tied_logits_matches_oracle(step):
    """Logits on a coarse grid: the k-th largest score sits in a run of exact
    ties in most rows, so the top-k threshold is settled either by keeping a
    radix bin whole (the select stops early) or by ranking the tied keys by
    index. The kept set has no rounding to hide behind: codes must match the
    oracle except where the Gumbel-perturbed winner or the top-p mass is a
    near tie."""
    V, rows, group = 2048, 256, 5
    rng = np.random.default_rng(int(1 / step))
    lg = (np.round(rng.standard_normal((rows, V)) * 0.8 / step) * step).astype(np.float32)
    samp = dict(
        temperature=rng.choice([0.7, 1.0], size=rows).astype(np.float32),
        top_k=rng.choice([1, 2, 5, 17, 50, 64, 100, 1000], size=rows).astype(np.int32),
        top_p=rng.choice([1.0, 0.9, 0.6], size=rows).astype(np.float32),
        seed=rng.integers(0, 2 ** 63, size=rows, dtype=np.int64).astype(np.uint64),
        offset=rng.integers(0, 2 ** 40, size=rows, dtype=np.int64))
    codes = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
    cp.test_draw(torch.from_numpy(lg).cuda(), torch_io.sampler_to_torch(samp), group, codes)
    got = codes.cpu().numpy()
    mism = 0
    for r in range(rows):
        d = oracle.draw_detail(lg[r], samp["temperature"][r], samp["top_k"][r], samp["top_p"][r],
                               int(samp["seed"][r]), r, int(samp["offset"][r]) + group)
        if d["code"] != got[r]:
            assert d["margin"] < 1e-4 or d["topp_gap"] < 1e-5, (r, got[r], d)
            mism += 1
    assert mism <= 2


# ---------------------------------------------------------------- frames
@pytest.mark.parametrize("kind", ["greedy", "mixed"])
def test_tiny_frame_matches_oracle(kind):
    fr = helpers.handle("tiny")
    s = fr.shape
    h, c0, samp = helpers.inputs("tiny", 5, kind, seed=1)
    gpu = helpers.run_gpu(fr, s, h, c0, samp)
    st = helpers.compare("tiny", h, c0, samp, gpu)
    print(f"tiny R=5 {kind}", st)
    assert st["near_ties"] <= 1, st


def test_tiny_frame_one_row_config():
    """The tiny decoder at 1 row, greedy, seed 0."""
    fr = helpers.handle("tiny")
    h, c0, samp = helpers.inputs("tiny", 1, "greedy", seed=0)
    gpu = helpers.run_gpu(fr, fr.shape, h, c0, samp)
    print("tiny R=1 greedy", helpers.compare("tiny", h, c0, samp, gpu))


def test_full_frame_one_row_greedy():
    fr = helpers.handle("full")
    h, c0, samp = helpers.inputs("full", 1, "greedy", seed=0)
    gpu = helpers.run_gpu(fr, fr.shape, h, c0, samp)
    st = helpers.compare("full", h, c0, samp, gpu)
    print("full R=1 greedy", st)


def test_full_frame_64_rows_sampled():
    """64 rows, temperature 0.9, top-k 50, top-p 0.8, seed = row, offset 0."""
    fr = helpers.handle("full")
    h, c0, samp = helpers.inputs("full", 64, "fixed", seed=0)
    gpu = helpers.run_gpu(fr, fr.shape, h, c0, samp)
    st = helpers.compare("full", h, c0, samp, gpu)
    print("full R=64 sampled", st)
    assert st["near_ties"] <= 0.05 * 64 * 15, st


@pytest.mark.parametrize("rows", [13, 59])
def test_full_frame_mixed_rows(rows):
    fr = helpers.handle("full")
    h, c0, samp = helpers.inputs("full", rows, "mixed", seed=3)
    gpu = helpers.run_gpu(fr, fr.shape, h, c0, samp)
    st = helpers.compare("full", h, c0, samp, gpu, seed=0)
    print(f"full R={rows} mixed", st)


# ---------------------------------------------------------------- 128-row frames
def test_full_frame_128_rows_sampled():
    """128 rows (M = 128 projections), temperature 0.9, top-k 50, top-p 0.8,
    seed = row, offset 0."""
    fr = helpers.handle("full_r128")
    assert fr.info.specialized == 1
    h, c0, samp = helpers.inputs("full", 128, "fixed", seed=0)
    gpu = helpers.run_gpu(fr, fr.shape, h, c0, samp)
    st = helpers.compare("full", h, c0, samp, gpu)
    print("full R=128 sampled", st)


@pytest.mark.parametrize("rows", [65, 100])
def test_full_frame_over_64_rows_mixed(rows):
    fr = helpers.handle("full_r128")
    h, c0, samp = helpers.inputs("full", rows, "mixed", seed=15)
    gpu = helpers.run_gpu(fr, fr.shape, h, c0, samp)
    st = helpers.compare("full", h, c0, samp, gpu)
    print(f"full R={rows} mixed (128-row handle)", st)


def test_tiny_frame_128_rows_generic_build():
    """The shape-generic build with M = 128 projections."""
    fr = helpers.handle("tiny_r128")
    assert fr.info.specialized == 0
    h, c0, samp = helpers.inputs("tiny", 128, "mixed", seed=16)
    gpu = helpers.run_gpu(fr, fr.shape, h, c0, samp)
    st = helpers.compare("tiny", h, c0, samp, gpu)
    print("tiny R=128 mixed", st)


def test_128_row_handle_invariants():
    """A 128-row handle: a second run, the per-phase graph, and the first 16
    rows run alone give the same bits; and its rows agree bit for bit with
    a 64-row handle's (the M = 128 and M = 64 tiles add the same products in
    the same order)."""
    fr = helpers.handle("full_r128")
    s = fr.shape
    h, c0, samp = helpers.inputs("full", 128, "mixed", seed=17)
    a = helpers.run_gpu(fr, s, h, c0, samp)
    for x in (helpers.run_gpu(fr, s, h, c0, samp), helpers.run_gpu(fr, s, h, c0, samp, split=True)):
        assert x["status"] == 0
        for k in ("codes", "logits", "emb_sum", "offset"):
            np.testing.assert_array_equal(a[k], x[k], err_msg=k)
    sub = {k: v[:16].copy() for k, v in samp.items()}
    b = helpers.run_gpu(fr, s, h[:16].copy(), c0[:16].copy(), sub)
    c = helpers.run_gpu(helpers.handle("full"), helpers.synth.shape("full"), h[:16].copy(), c0[:16].copy(), sub)
    for x in (b, c):
        np.testing.assert_array_equal(a["codes"][:16], x["codes"])
        np.testing.assert_array_equal(a["logits"][:, :16], x["logits"])
        np.testing.assert_array_equal(a["emb_sum"][:16], x["emb_sum"])


# ---------------------------------------------------------------- per-chunk waits
@pytest.mark.parametrize("name,rows,max_ctas", [("full", 64, 0), ("full_r128", 128, 0), ("tiny", 37, 0),
                                                ("full", 24, 64)])
def test_chunk_waits_give_the_same_bits(name, rows, max_ctas):
    """Per-chunk waits (the default) change only when each input chunk is
    staged, not what any tile adds or in which order: codes, logits,
    embedding sums and offsets are bit-identical to whole-phase waits, and to
    the per-phase graph (with 64 CTAs, two-tile tasks signal a counter per
    tile)."""
    base = helpers.handle(name, max_ctas=max_ctas, phase_waits=True)
    ch = helpers.handle(name, max_ctas=max_ctas)
    s = base.shape
    h, c0, samp = helpers.inputs(name, rows, "mixed", seed=18)
    a = helpers.run_gpu(base, s, h, c0, samp)
    for x in (helpers.run_gpu(ch, s, h, c0, samp), helpers.run_gpu(ch, s, h, c0, samp),
              helpers.run_gpu(ch, s, h, c0, samp, split=True)):
        assert x["status"] == 0
        for k in ("codes", "logits", "emb_sum", "offset"):
            np.testing.assert_array_equal(a[k], x[k], err_msg=k)


def test_phase_waits_timeout_is_reported_not_hung():
    """The timeout path with whole-phase waits (the default per-chunk waits
    are exercised by the other abort tests): the frame ends with
    CP_ERR_TIMEOUT and the handle runs again once cleared."""
    s = helpers.synth.shape("tiny")
    fr = helpers.handle("tiny", debug_stall_task=3, timeout_ns=50_000_000, phase_waits=True)
    h, c0, samp = helpers.inputs("tiny", 2, "greedy", seed=0)
    out = helpers.run_gpu(fr, s, h, c0, samp, want_logits=False)
    assert out["status"] == cp.CP_ERR_TIMEOUT
    fr.clear_status()
    assert fr.status() == 0


# ---------------------------------------------------------------- invariants
def test_bit_identical_runs_and_split_graph():
    fr = helpers.handle("full")
    s = fr.shape
    h, c0, samp = helpers.inputs("full", 64, "mixed", seed=4)
    a = helpers.run_gpu(fr, s, h, c0, samp)
    b = helpers.run_gpu(fr, s, h, c0, samp)
    c = helpers.run_gpu(fr, s, h, c0, samp, split=True)
    d = helpers.run_gpu(fr, s, h, c0, samp, split=True)
    for x in (b, c, d):
        assert x["status"] == 0
        for k in ("codes", "logits", "emb_sum", "offset"):
            np.testing.assert_array_equal(a[k], x[k], err_msg=k)


def test_specialized_build_matches_generic_build():
    """The full shape runs the frame kernel build with its sizes fixed at
    compile time; the build that reads every size at run time must give the
    same bits (same tiles, same sums in the same order), through cp_frame and
    through the per-phase graph."""
    fr = helpers.handle("full")
    gen = helpers.handle("full", generic_kernel=True)
    assert fr.info.specialized == 1 and gen.info.specialized == 0
    assert helpers.handle("tiny").info.specialized == 0
    s = fr.shape
    h, c0, samp = helpers.inputs("full", 59, "mixed", seed=9)
    a = helpers.run_gpu(fr, s, h, c0, samp)
    b = helpers.run_gpu(gen, s, h, c0, samp)
    c = helpers.run_gpu(gen, s, h, c0, samp, split=True)
    for x in (a, b, c):
        assert x["status"] == 0
    for x in (b, c):
        for k in ("codes", "logits", "emb_sum", "offset"):
            np.testing.assert_array_equal(a[k], x[k], err_msg=k)


def test_rows_independent_of_batch():
    fr = helpers.handle("full")
    s = fr.shape
    h, c0, samp = helpers.inputs("full", 64, "mixed", seed=6)
    a = helpers.run_gpu(fr, s, h, c0, samp)
    sub = {k: v[:16].copy() for k, v in samp.items()}
    b = helpers.run_gpu(fr, s, h[:16].copy(), c0[:16].copy(), sub)
    np.testing.assert_array_equal(a["codes"][:16], b["codes"])
    np.testing.assert_array_equal(a["logits"][:, :16], b["logits"])
    np.testing.assert_array_equal(a["emb_sum"][:16], b["emb_sum"])


def test_frames_chain_on_device():
    """Frame f+1 takes frame f's last code as its first code and carries the
    offsets, with no host round trip between frames."""
    fr = helpers.handle("tiny")
    s = fr.shape
    R, P = 8, s["positions"]
    h, c0, samp = helpers.inputs("tiny", R, "mixed", seed=2)
    ts = torch_io.sampler_to_torch(samp)
    tc = torch.from_numpy(c0).cuda()
    codes = torch.zeros((R, P - 1), dtype=torch.int32, device="cuda")
    for f in range(3):
        hf = torch.from_numpy(helpers.synth.talker_hidden(s, R, 2, frame=f)).cuda()
        fr.frame(hf, tc, ts, R, codes)
        tc = codes[:, -1].contiguous()
    torch.cuda.synchronize()
    assert fr.status() == 0
    np.testing.assert_array_equal(ts["offset"].cpu().numpy(), 3 * (P - 1))


def test_chained_frames_match_oracle():
    """The row-sweep workload's chaining (mixed per-row samplers, 16 rows):
    three frames back to back on the device, each taking the previous frame's
    last code as its first code and the offsets it advanced, with a fresh
    talker hidden state per frame and no host round trip between them. Every
    frame's codes and logits are then checked against the oracle run on the
    same carried inputs."""
    fr = helpers.handle("full")
    s = fr.shape
    R, P, V, H = 16, s["positions"], s["vocab"], s["hidden"]
    _, c0, samp = helpers.inputs("full", R, "mixed", seed=12)
    ts = torch_io.sampler_to_torch(samp)
    nf = 3
    hs = [helpers.synth.talker_hidden(s, R, 12, frame=f) for f in range(nf)]
    codes = torch.full((nf, R, P - 1), -1, dtype=torch.int32, device="cuda")
    es = torch.zeros((nf, R, H), dtype=torch.float32, device="cuda")
    lg = torch.empty((nf, P - 1, R, V), dtype=torch.float32, device="cuda")
    offs = torch.empty((nf, R), dtype=torch.int64, device="cuda")
    hd = [torch.from_numpy(x).cuda() for x in hs]
    torch.cuda.synchronize()
    tc = torch.from_numpy(c0).cuda()
    for f in range(nf):
        fr.frame(hd[f], tc, ts, R, codes[f], es[f])
        offs[f].copy_(ts["offset"])
        for j in range(P - 1):
            fr.debug_logits(j, lg[f, j])
        tc = codes[f, :, -1].contiguous()
    torch.cuda.synchronize()
    assert fr.status() == 0
    cn, en, ln, on = codes.cpu().numpy(), es.cpu().numpy(), lg.cpu().numpy(), offs.cpu().numpy()
    first = c0
    for f in range(nf):
        sf = dict(samp, offset=np.asarray(samp["offset"]) + f * (P - 1))
        gpu = dict(codes=cn[f], emb_sum=en[f], logits=ln[f], status=0, offset=on[f])
        st = helpers.compare("full", hs[f], first, sf, gpu)
        print(f"chained frame {f}, R={R} mixed", st)
        first = cn[f][:, -1].copy()


def _cut_phases(s, kinds):
    """Phase indices (the oracle's phase order) at which a frame is cut: the
    first phase of each layer (qkv) and, for the attention/MLP composition,
    each layer's gate/up phase too."""
    return [i for i, ph in enumerate(oracle.plan.phases(s)) if ph[0] in kinds]


def test_cut_compositions_full_shape_bit_identical():
    """The cut-composition workload at 64 rows on the full shape: the frame as
    one launch, as one launch per layer (81), as attention-phase and
    MLP-phase launches (161) and as the per-phase graph gives the same bits
    (the same tiles add the same partial sums in the same order; counters
    persist across the launches)."""
    s = helpers.synth.shape("full")
    fr = helpers.handle("full")
    per_layer = _cut_phases(s, ("QKV",))
    attn_mlp = _cut_phases(s, ("QKV", "GU"))
    assert len(per_layer) == 80 and len(attn_mlp) == 160
    h, c0, samp = helpers.inputs("full", 64, "mixed", seed=14)
    a = helpers.run_gpu(fr, s, h, c0, samp)
    variants = [helpers.run_gpu(fr, s, h, c0, samp, split=True)]
    for cuts in (per_layer, attn_mlp):
        cut = helpers.handle("full", cuts=tuple(cuts))
        variants.append(helpers.run_gpu(cut, s, h, c0, samp))
    for x in variants:
        assert x["status"] == 0
        for k in ("codes", "logits", "emb_sum", "offset"):
            np.testing.assert_array_equal(a[k], x[k], err_msg=k)


@pytest.mark.parametrize("name,rows,cuts", [("tiny", 4, (2, 7, 16)), ("full_r128", 128, (27, 54, 200, 431))])
def test_cut_launches_match_single_launch(name, rows, cuts):
    s = helpers.synth.shape(name)
    fr = helpers.handle(name)
    cut = helpers.handle(name, cuts=cuts)
    h, c0, samp = helpers.inputs(name, rows, "mixed", seed=8)
    a = helpers.run_gpu(fr, s, h, c0, samp)
    b = helpers.run_gpu(cut, s, h, c0, samp)
    for k in ("codes", "logits", "emb_sum"):
        np.testing.assert_array_equal(a[k], b[k])


def test_timeout_is_reported_not_hung():
    """A wait that nothing satisfies ends the frame with CP_ERR_TIMEOUT after
    the handle's limit; the status is sticky until cleared; frames work again."""
    s = helpers.synth.shape("tiny")
    fr = helpers.handle("tiny", debug_stall_task=3, timeout_ns=50_000_000)
    h, c0, samp = helpers.inputs("tiny", 2, "greedy", seed=0)
    out = helpers.run_gpu(fr, s, h, c0, samp, want_logits=False)
    assert out["status"] == cp.CP_ERR_TIMEOUT
    assert fr.status() == cp.CP_ERR_TIMEOUT
    fr.clear_status()
    assert fr.status() == 0


def test_staging_abort_is_reported_not_hung():
    """The leader alone waits (for a count nothing sets) while staging a K
    part; its warp-mates must follow it through the abort instead of
    meeting it at a different warp-synchronous point. The frame ends with
    CP_ERR_TIMEOUT after the handle's limit, and the next frame, once the
    status is cleared, runs and matches the oracle."""
    s = helpers.synth.shape("tiny")
    fr = helpers.handle("tiny", debug_stall_staging=True, timeout_ns=50_000_000)
    h, c0, samp = helpers.inputs("tiny", 3, "greedy", seed=0)
    out = helpers.run_gpu(fr, s, h, c0, samp, want_logits=False)
    assert out["status"] == cp.CP_ERR_TIMEOUT
    fr.clear_status()
    assert fr.status() == 0


def test_attention_abort_after_early_copy_is_reported_not_hung():
    """An attention task past position 0 copies the earlier positions' keys
    and values (its own warp, before the leader's dependency wait). If that
    wait then gives up, the leader still completes the copy's barrier phase
    so the teardown drain finds it landed: the frame ends with CP_ERR_TIMEOUT,
    and a frame on a clean handle afterwards is bit-identical to the one
    traced before. With 16 CTAs every CTA holds an attention task of each
    position; the stalled one is CTA 0's at the last position, found from a
    traced frame (word 7 packs phase, kind and CTA)."""
    s = helpers.synth.shape("tiny")
    h, c0, samp = helpers.inputs("tiny", 64, "mixed", seed=4)
    tr = helpers.handle("tiny", max_ctas=16, trace=True)
    ref = helpers.run_gpu(tr, s, h, c0, samp, want_logits=False)
    t = torch.zeros((tr.info.tasks, 16), dtype=torch.int64, device="cuda")
    tr.trace(t)
    w7 = t[:, 7].cpu().numpy()
    phase, kind, cta = w7 >> 32, (w7 >> 16) & 0xFFFF, w7 & 0xFFFF
    mine = np.flatnonzero(cta == 0)
    assert mine.size and mine[0] == 0 and np.all(np.diff(mine) == 1)
    attn = mine[kind[mine] == 3]
    assert attn.size >= s["positions"]
    k = int(attn[np.argmax(phase[attn])]) + 1  # 1-based, in CTA 0's list
    fr = helpers.handle("tiny", max_ctas=16, debug_stall_task=k, timeout_ns=50_000_000)
    out = helpers.run_gpu(fr, s, h, c0, samp, want_logits=False)
    assert out["status"] == cp.CP_ERR_TIMEOUT
    fr.clear_status()
    again = helpers.run_gpu(helpers.handle("tiny", max_ctas=16), s, h, c0, samp, want_logits=False)
    for k2 in ("codes", "emb_sum"):
        np.testing.assert_array_equal(again[k2], ref[k2], err_msg=k2)


def test_range_error_is_reported_not_hung():
    """The normed projections' partial sums travel between the cluster's CTAs
    as fp16 after the norm's row factor. Attention-norm gains of about 1e6
    push the qkv partials (then ~1e5) outside the fp16 range: the frame stops
    with the sticky CP_ERR_RANGE within its wait limit, without a fault, and
    the status clears."""
    s = helpers.synth.shape("tiny")
    w = dict(helpers.synth.weights(s, 0))
    w["attn_norm"] = np.full_like(w["attn_norm"], 0x4974)  # bf16 999424
    fr = cp.Frame(s, torch_io.weights_to_torch(w), timeout_ns=50_000_000)
    try:
        h, c0, samp = helpers.inputs("tiny", 4, "mixed", seed=0)
        out = helpers.run_gpu(fr, s, h, c0, samp, want_logits=False)
        assert out["status"] == cp.CP_ERR_RANGE
        assert fr.status() == cp.CP_ERR_RANGE   # sticky
        fr.clear_status()
        assert fr.status() == 0
    finally:
        fr.close()


@pytest.mark.parametrize("name,rows", [("full", 24), ("full_r128", 72)])
def test_results_independent_of_grid(name, rows):
    """A smaller grid (16 clusters) puts two tiles on one cluster in the qkv,
    gate/up and head phases (a 128-row handle runs them as second rounds
    instead) and runs extra rounds elsewhere; every tile still adds the same
    K parts in the same order, so results are bit-identical."""
    s = helpers.synth.shape(name)
    fr = helpers.handle(name)
    small = helpers.handle(name, max_ctas=64)
    assert small.info.grid == 64
    h, c0, samp = helpers.inputs(name, rows, "mixed", seed=9)
    a = helpers.run_gpu(fr, s, h, c0, samp)
    b = helpers.run_gpu(small, s, h, c0, samp)
    for k in ("codes", "logits", "emb_sum", "offset"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


def test_keys_and_values_match_oracle():
    """The keys (after QK-Norm and RoPE) and values each layer wrote at each
    position, read back through cp_debug_state, against the float64 oracle
    teacher-forced at the GPU's codes. These are intermediates: relative L2
    error within the logits' 1e-2 per layer and position, and every value
    within twice the logit tolerance plus one bf16 ulp of itself (they are
    stored as bf16, so upstream float error can move that last rounding by a
    whole ulp; QK-Norm turns the relative error of q/k into absolute error at
    unit scale, and the error of earlier layers reaches the later ones)."""
    fr = helpers.handle("full")
    s = fr.shape
    R = 13
    h, c0, samp = helpers.inputs("full", R, "mixed", seed=5)
    gpu = helpers.run_gpu(fr, s, h, c0, samp)
    _, _, W = helpers.model("full", 0)
    ref = oracle.run_frame(s, W, h, c0, samp, "fp64", forced_codes=gpu["codes"], keep_kv=True)
    Hkv, D = s["kv_heads"], s["head_dim"]
    buf = torch.zeros((R, Hkv, D), dtype=torch.int16, device="cuda")
    for what, key in ((1, "K"), (2, "V")):
        for l in range(s["layers"]):
            for pos in range(s["positions"]):
                fr.debug_state(what, l, pos, buf)
                torch.cuda.synchronize()
                got = helpers.synth.bf16_bits_to_f32(buf.cpu().numpy().view(np.uint16)).astype(np.float64)
                want = ref[key][l, pos]
                excess = np.abs(got - want) - (2 * helpers.LOGIT_TOL + np.abs(want) * 2.0 ** -8)
                assert excess.max() <= 0, (key, l, pos, float(np.abs(got - want).max()))
                rel = np.linalg.norm(got - want) / np.linalg.norm(want)
                assert rel <= helpers.REL_L2_TOL, (key, l, pos, rel)


@pytest.mark.parametrize("rows", [2, 24])
def test_wide_frame_matches_oracle(rows):
    """The 2x-wide decoder (hidden 2048, 16 q and 16 kv heads, FFN 6144):
    longer K parts (8 chunks for qkv and gate/up, 24 for down, through 8 A
    slots), two-tile qkv tasks (48 tiles on 36 clusters), 16 kv groups of one
    q head, 64 gate/up tiles signalling one counter each; mixed sampling."""
    fr = helpers.handle("wide")
    h, c0, samp = helpers.inputs("wide", rows, "mixed", seed=11)
    gpu = helpers.run_gpu(fr, fr.shape, h, c0, samp)
    st = helpers.compare("wide", h, c0, samp, gpu)
    print(f"wide R={rows} mixed", st)
