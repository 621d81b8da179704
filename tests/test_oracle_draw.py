"""Pins for the oracle's Philox stream and draw (CPU only)."""
import os

import numpy as np
import pytest

from oracle import philox
from oracle.draw import draw, draw_detail


# ---------------------------------------------------------------- Philox
def _triton_philox(seed, ctr):
    """Philox4x32-10 as implemented by triton, run under its CPU interpreter."""
    os.environ["TRITON_INTERPRET"] = "1"
    triton = pytest.importorskip("triton")
    import triton.language as tl
    import torch

    @triton.jit
    def k(out_ptr, seed, cp, N: tl.constexpr):
        o = tl.arange(0, N)
        c0 = tl.load(cp + o * 4 + 0).to(tl.uint32, bitcast=True)
        c1 = tl.load(cp + o * 4 + 1).to(tl.uint32, bitcast=True)
        c2 = tl.load(cp + o * 4 + 2).to(tl.uint32, bitcast=True)
        c3 = tl.load(cp + o * 4 + 3).to(tl.uint32, bitcast=True)
        a, b, c, d = tl.philox(seed, c0, c1, c2, c3)
        tl.store(out_ptr + o * 4 + 0, a.to(tl.int32, bitcast=True))
        tl.store(out_ptr + o * 4 + 1, b.to(tl.int32, bitcast=True))
        tl.store(out_ptr + o * 4 + 2, c.to(tl.int32, bitcast=True))
        tl.store(out_ptr + o * 4 + 3, d.to(tl.int32, bitcast=True))

    n = ctr.shape[0]
    out = torch.zeros(n * 4, dtype=torch.int32)
    k[(1,)](out, seed, torch.from_numpy(ctr.astype(np.uint32).view(np.int32).reshape(-1).copy()), N=n)
    return out.numpy().view(np.uint32).reshape(n, 4)


@pytest.mark.parametrize("seed", [0, 1, 0x123456789ABCDEF0, (1 << 64) - 1])
def test_philox_matches_triton(seed):
    rng = np.random.default_rng(11)
    ctr = rng.integers(0, 2 ** 32, size=(64, 4), dtype=np.uint64)
    ctr[0] = 0
    ctr[1] = 0xFFFFFFFF
    want = _triton_philox(seed, ctr)
    got = np.stack(philox.philox4x32(tuple(ctr.T), (seed & 0xFFFFFFFF, seed >> 32)), axis=1)
    np.testing.assert_array_equal(got, want)


def test_philox_words_look_uniform():
    w = philox.vocab_words(seed=7, row=3, offset=11, vocab=1 << 16)
    bits = ((w[:, None] >> np.arange(32, dtype=np.uint32)) & 1).mean(axis=0)
    assert np.all(np.abs(bits - 0.5) < 0.01)
    assert len(np.unique(w)) > 65000


def test_uniform_mapping_is_open_interval_and_exact():
    u = philox.uniform_from_word(np.array([0, 511, 512, 0xFFFFFFFF], dtype=np.uint32))
    assert u[0] == np.float32(2.0 ** -24) and u[1] == u[0]
    assert u[2] == np.float32(3 * 2.0 ** -24)
    assert float(u[3]) == 1 - 2.0 ** -24 and u[3] < 1
    # every one of the 2^23 values is distinct, so the map loses nothing to rounding
    k = np.arange(0, 1 << 23, dtype=np.uint32) << np.uint32(9)
    assert np.unique(philox.uniform_from_word(k)).size == 1 << 23
    assert np.all(np.isfinite(-np.log(-np.log(philox.uniform_from_word(k)))))


def test_stream_changes_with_seed_row_offset():
    base = philox.vocab_words(1, 2, 3, 256)
    for args in ((2, 2, 3), (1, 3, 3), (1, 2, 4), (1, 2, 3 + (1 << 32))):
        assert np.mean(philox.vocab_words(*args, 256) == base) < 0.02


def test_vocab_word_layout():
    # entry v reads word v & 3 of the block at counter v >> 2
    seed, row, off = 5, 9, (7 << 32) | 3
    words = philox.vocab_words(seed, row, off, 16)
    blk = philox.philox4x32((np.uint64(2), row, 3, 7), (5, 0))
    assert [int(words[8 + i]) for i in range(4)] == [int(b) for b in blk]


# ---------------------------------------------------------------- draw
def _logits(V, seed):
    return (np.random.default_rng(seed).standard_normal(V) * 0.6).astype(np.float32)


def test_temperature_zero_is_argmax_lowest_index():
    lg = _logits(256, 1)
    assert draw(lg, 0.0, 0, 1.0, 0, 0, 0) == int(np.argmax(lg))
    lg[10] = lg[200] = lg.max() + 1
    assert draw(lg, 0.0, 50, 0.5, 9, 1, 2) == 10


def test_top_k_one_is_argmax_for_any_seed():
    lg = _logits(512, 2)
    for seed in range(20):
        assert draw(lg, 0.9, 1, 1.0, seed, 0, seed * 3) == int(np.argmax(lg))


def test_tiny_top_p_is_argmax():
    lg = _logits(512, 3)
    for seed in range(20):
        assert draw(lg, 1.3, 0, 1e-6, seed, 1, 0) == int(np.argmax(lg))


def _frequencies(lg, T, k, p, n):
    V = lg.shape[0]
    cnt = np.zeros(V)
    for off in range(n):
        cnt[draw(lg, T, k, p, 42, 0, off)] += 1
    return cnt


def _chi2_ok(cnt, prob):
    n = cnt.sum()
    m = prob > 0
    assert cnt[~m].sum() == 0
    exp = n * prob[m]
    chi2 = ((cnt[m] - exp) ** 2 / exp).sum()
    dof = m.sum() - 1
    # 5-sigma bound on a chi-square with dof degrees of freedom
    return chi2 < dof + 5 * np.sqrt(2 * dof)


@pytest.mark.slow
def test_unfiltered_draw_frequencies_follow_softmax():
    lg = np.array([0.3, -0.2, 1.1, 0.0, -1.0, 0.7, 0.2, -0.5], np.float32)
    T = 0.8
    prob = np.exp(lg / T)
    prob /= prob.sum()
    assert _chi2_ok(_frequencies(lg, T, 0, 1.0, 20000), prob)


@pytest.mark.slow
def test_top_k_draw_frequencies_follow_renormalised_softmax():
    lg = np.array([0.3, -0.2, 1.1, 0.0, -1.0, 0.7, 0.2, -0.5], np.float32)
    T, k = 1.1, 3
    top = np.argsort(-lg)[:k]
    prob = np.zeros(8)
    prob[top] = np.exp(lg[top] / T)
    prob /= prob.sum()
    assert _chi2_ok(_frequencies(lg, T, k, 1.0, 20000), prob)


@pytest.mark.slow
def test_top_p_support_and_frequencies():
    lg = np.array([2.0, 1.0, 0.5, 0.0, -0.5, -3.0], np.float32)
    T, p = 1.0, 0.8
    pr = np.exp(lg - lg.max())
    pr /= pr.sum()
    before = np.concatenate([[0], np.cumsum(pr)[:-1]])
    keep = before < p                         # logits are already in descending order
    prob = np.where(keep, pr, 0)
    prob /= prob.sum()
    assert keep.sum() == 3
    assert _chi2_ok(_frequencies(lg, T, 0, p, 20000), prob)


def test_top_k_tie_break_by_index():
    lg = np.zeros(16, np.float32)
    lg[[3, 7, 12]] = 1.0                       # three-way tie for first
    for off in range(40):
        c = draw(lg, 1.0, 2, 1.0, 1, 0, off)
        assert c in (3, 7)                     # k = 2 keeps the two lowest indices of the tie


def test_margin_reports_gap():
    lg = np.array([1.0, 0.5, 0.25], np.float32)
    d = draw_detail(lg, 0.0, 0, 1.0, 0, 0, 0)
    assert d["code"] == 0 and abs(d["margin"] - 0.5) < 1e-7


def test_topp_band_bounds_the_mass_move_of_a_logit_perturbation():
    """The near-tie band for top-p boundaries: logits moved by at most delta
    move the softmax mass before any token (in the unperturbed order) by no
    more than the band, at every temperature. The extreme move comes from
    +delta on the tokens before k and -delta on the rest (or the reverse);
    for small masses it nearly reaches the band, so a band built on
    exp(delta / T) instead of exp(2 delta / T) fails here."""
    import helpers
    rng = np.random.default_rng(11)
    worst_ratio = 0.0
    for trial in range(200):
        V = int(rng.choice([8, 64, 512]))
        T = float(rng.choice([0.05, 0.1, 0.4, 0.9, 1.2]))
        delta = float(rng.choice([1e-3, 1e-2, 3e-2]))
        lg = rng.standard_normal(V) * rng.choice([0.5, 2.0])
        order = np.argsort(-lg, kind="stable")

        def mass_before(x):
            pr = np.exp((x - x.max()) / T)
            pr /= pr.sum()
            return np.concatenate([[0.0], np.cumsum(pr[order])[:-1]])

        m0 = mass_before(lg)
        for k in rng.integers(1, V, size=8):
            before = np.zeros(V, bool)
            before[order[:k]] = True
            for sign in (1.0, -1.0):
                pert = lg + np.where(before, sign * delta, -sign * delta)
                moved = abs(mass_before(pert)[k] - m0[k])
                allowed = helpers.topp_band(m0[k], 0.0, delta, T, delta) - helpers.TOPP_TOL
                assert moved <= allowed * (1 + 1e-9) + 1e-15, (trial, k, moved, allowed)
                if allowed > 1e-6:
                    worst_ratio = max(worst_ratio, moved / allowed)
            pert = lg + rng.uniform(-delta, delta, V)
            assert abs(mass_before(pert)[k] - m0[k]) <= helpers.topp_band(m0[k], 0.0, delta, T, delta)
    assert worst_ratio > 0.9  # the bound is nearly reached: it is not loose by a factor
    # the band never follows a logit difference past the stated tolerance
    assert helpers.topp_band(0.8, 0.0, 1.0, 0.5, 3e-2) == helpers.topp_band(0.8, 0.0, 3e-2, 0.5, 3e-2)
