"""Pins for the oracle's elementary operations (CPU only).

Each check ties an oracle function to something other than itself: values
worked out by hand, closed forms, invariants, or a library routine.
"""
import math

import numpy as np
import pytest
import torch

from oracle.frame import attention, bf16_round, rms_norm, rope, silu


# ---------------------------------------------------------------- bf16 rounding
def test_bf16_round_hand_values():
    # 1 + 2^-8 lies half way between 1 and 1 + 2^-7: ties go to the even one (1).
    # 1 + 3*2^-8 lies half way between 1 + 2^-7 and 1 + 2^-6: even is 1 + 2^-6.
    vals = np.array([1.0, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -20,
                     -2.5, 3.0e-3, 65504.0])
    want = np.array([1.0, 1.0, 1 + 2.0 ** -6, 1 + 2.0 ** -7, -2.5, None, None], dtype=object)
    got = bf16_round(vals)
    for g, w in zip(got[:5], want[:5]):
        assert g == w
    # every result has at most 8 significant bits
    m, _ = np.frexp(got)
    assert np.all((m * 2 ** 8) == np.round(m * 2 ** 8))


def test_bf16_round_matches_torch_on_float32_values():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-20, 20, 100000))).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(bf16_round(x.astype(np.float64)), want)


# ---------------------------------------------------------------- RMSNorm
def test_rms_norm_hand_value():
    # mean(3^2, 4^2) = 12.5, sqrt = 3.5355...; [3, 4] / 3.5355 = [0.8485, 1.1314]
    got = rms_norm(np.array([3.0, 4.0]), np.ones(2), 0.0)
    np.testing.assert_allclose(got, [0.848528137423857, 1.131370849898476], rtol=1e-14)


def test_rms_norm_matches_torch():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((5, 64))
    g = 1 + 0.01 * rng.standard_normal(64)
    want = torch.nn.functional.rms_norm(torch.from_numpy(v), (64,), torch.from_numpy(g), eps=1e-6)
    np.testing.assert_allclose(rms_norm(v, g, 1e-6), want.numpy(), rtol=1e-12)


def test_rms_norm_scale_invariant():
    rng = np.random.default_rng(3)
    v = rng.standard_normal(32)
    np.testing.assert_allclose(rms_norm(v, 1.0, 0.0), rms_norm(7.5 * v, 1.0, 0.0), rtol=1e-13)


# ---------------------------------------------------------------- RoPE
def test_rope_position_zero_is_identity():
    v = np.random.default_rng(4).standard_normal((3, 128))
    np.testing.assert_array_equal(rope(v, 0, 10000.0), v)


def test_rope_preserves_norm_and_composes():
    v = np.random.default_rng(5).standard_normal(64)
    for p in (1, 5, 15):
        np.testing.assert_allclose(np.linalg.norm(rope(v, p, 1e4)), np.linalg.norm(v), rtol=1e-13)
    # rotating by positions a then b equals rotating by a + b
    np.testing.assert_allclose(rope(rope(v, 3, 1e4), 4, 1e4), rope(v, 7, 1e4), atol=1e-13)


@pytest.mark.parametrize("i", [0, 1, 17, 63])
def test_rope_one_pair_is_a_plane_rotation(i):
    D, p, base = 128, 9, 10000.0
    v = np.zeros(D)
    v[i], v[i + D // 2] = 0.6, -0.8
    ang = p * base ** (-2.0 * i / D)
    out = rope(v, p, base)
    want = np.zeros(D)
    want[i] = 0.6 * math.cos(ang) + 0.8 * math.sin(ang)
    want[i + D // 2] = -0.8 * math.cos(ang) + 0.6 * math.sin(ang)
    np.testing.assert_allclose(out, want, atol=1e-15)


# ---------------------------------------------------------------- SiLU
def test_silu_values():
    assert silu(0.0) == 0.0
    assert abs(silu(40.0) - 40.0) < 1e-12
    assert abs(silu(-40.0)) < 1e-12
    np.testing.assert_allclose(silu(1.0), 1.0 / (1.0 + math.exp(-1.0)), rtol=1e-15)
    z = np.linspace(-8, 8, 101)
    np.testing.assert_allclose(silu(z), torch.nn.functional.silu(torch.from_numpy(z)).numpy(), rtol=1e-13)


# ---------------------------------------------------------------- attention
def _rand_qkv(T, R, Hq, Hkv, D, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((R, Hq, D)), rng.standard_normal((T, R, Hkv, D)),
            rng.standard_normal((T, R, Hkv, D)))


def test_attention_first_position_returns_v0():
    q, K, V = _rand_qkv(1, 2, 4, 2, 16, 6)
    out = attention(q, K, V)
    for h in range(4):
        np.testing.assert_allclose(out[:, h], V[0, :, h // 2], rtol=1e-15)


def test_attention_zero_query_averages_values():
    q, K, V = _rand_qkv(5, 1, 2, 1, 8, 7)
    out = attention(np.zeros_like(q), K, V)
    np.testing.assert_allclose(out[0, 0], V[:, 0, 0].mean(axis=0), rtol=1e-13)


def test_attention_brute_force_single_head():
    q, K, V = _rand_qkv(4, 1, 1, 1, 6, 8)
    scores = []
    for t in range(4):
        scores.append(sum(q[0, 0, d] * K[t, 0, 0, d] for d in range(6)) / math.sqrt(6))
    mx = max(scores)
    w = [math.exp(s - mx) for s in scores]
    z = sum(w)
    want = [sum(w[t] / z * V[t, 0, 0, d] for t in range(4)) for d in range(6)]
    np.testing.assert_allclose(attention(q, K, V)[0, 0], want, rtol=1e-13)


def test_attention_gqa_matches_torch_sdpa():
    T, R, Hq, Hkv, D = 6, 3, 8, 2, 16
    q, K, V = _rand_qkv(T, R, Hq, Hkv, D, 9)
    tq = torch.from_numpy(q)[:, :, None, :]                       # [R][Hq][1][D]
    tk = torch.from_numpy(K).permute(1, 2, 0, 3)                  # [R][Hkv][T][D]
    tv = torch.from_numpy(V).permute(1, 2, 0, 3)
    want = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, enable_gqa=True)
    np.testing.assert_allclose(attention(q, K, V), want[:, :, 0].numpy(), rtol=1e-12, atol=1e-13)


def test_attention_gqa_equals_mha_with_repeated_kv():
    T, R, Hq, Hkv, D = 3, 2, 4, 2, 8
    q, K, V = _rand_qkv(T, R, Hq, Hkv, D, 10)
    Kr, Vr = np.repeat(K, 2, axis=2), np.repeat(V, 2, axis=2)
    np.testing.assert_allclose(attention(q, K, V), attention(q, Kr, Vr), rtol=1e-14)
