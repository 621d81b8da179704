"""Pins for the oracle's whole frame (CPU only)."""
import json
import os

import numpy as np
import pytest
import torch

import synth
from oracle import plan, run_frame
from oracle.frame import Weights, rms_norm

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")


def _tiny(rows=2, kind="greedy", seed=0):
    s = synth.shape("tiny")
    w = synth.weights(s, seed)
    return s, w, synth.talker_hidden(s, rows, seed), synth.first_codes(s, rows, seed), \
        synth.sampler(kind, rows, seed)


# ---------------------------------------------------------------- closed forms
def test_phase_count_and_weight_bytes_match_the_pages():
    g = json.load(open(GOLDEN))
    s = synth.shape("full")
    ph = plan.phases(s)
    assert len(ph) == g["phases"] == 432
    assert sum(1 for k in ph if k[0] == "DRAW") == g["draws"]
    assert sum(1 for k in ph if k[0] == "HEAD") == g["heads"]
    assert sum(1 for k in ph if k[0] in ("EMB0", "DRAW")) == g["embedding_steps"]
    b = plan.weight_bytes(s)
    assert round(b["layers"] / 1e6) == g["layers_weight_MB"]
    assert abs(b["frame"] / 1e9 - g["frame_weight_GB_approx"]) < 0.05
    assert abs(b["frame"] / 4.8e12 * 1e3 - g["floor_ms_at_4p8_TBps"]) < 0.005
    assert b["frame"] == 2583691264 == synth.weight_bytes_per_frame(s)
    assert len(plan.phases(synth.shape("tiny"))) == 28


# ---------------------------------------------------------------- structure
def test_zero_attention_and_mlp_outputs_leave_the_residual():
    """With w_o = w_down = 0 every position's output is its input, so head j
    sees table j's embedding of code j: the head/table indexing in closed form."""
    s, w, h, c0, sp = _tiny(rows=3)
    w = dict(w)
    w["w_o"] = np.zeros_like(w["w_o"])
    w["w_down"] = np.zeros_like(w["w_down"])
    out = run_frame(s, w, h, c0, sp, "fp64")
    W = Weights(w)
    codes = np.concatenate([c0[:, None], out["codes"]], axis=1)
    for j in range(s["positions"] - 1):
        x = W["embed"][j][codes[:, j]]
        want = rms_norm(x, W["final_norm"], s["rms_eps"]) @ W["heads"][j].T
        np.testing.assert_allclose(out["logits"][j], want, rtol=1e-12, atol=1e-14)
        assert np.array_equal(out["codes"][:, j], np.argmax(want, axis=1))


def test_teacher_forcing_with_own_codes_is_identity():
    s, w, h, c0, sp = _tiny(rows=3, kind="mixed")
    a = run_frame(s, w, h, c0, sp, "bf16io")
    b = run_frame(s, w, h, c0, sp, "bf16io", forced_codes=a["codes"])
    np.testing.assert_array_equal(a["logits"], b["logits"])
    np.testing.assert_array_equal(a["codes"], b["drawn"])


def test_rows_are_independent():
    s, w, h, c0, sp = _tiny(rows=4, kind="mixed")
    full = run_frame(s, w, h, c0, sp, "fp64")
    one = run_frame(s, w, h[:1], c0[:1], {k: v[:1] for k, v in sp.items()}, "fp64")
    np.testing.assert_allclose(full["logits"][:, :1], one["logits"], rtol=1e-10, atol=1e-13)
    np.testing.assert_array_equal(full["codes"][:1], one["codes"])


def test_offsets_advance_by_groups_for_every_row_and_emb_sum():
    s, w, h, c0, sp = _tiny(rows=3, kind="mixed")
    sp["offset"] = np.array([0, 5, 1 << 40], np.int64)
    sp["temperature"][1] = 0.0
    out = run_frame(s, w, h, c0, sp, "fp64")
    np.testing.assert_array_equal(out["offset"], sp["offset"] + s["positions"] - 1)
    W = Weights(w)
    codes = np.concatenate([c0[:, None], out["codes"]], axis=1)
    want = sum(W["embed"][k][codes[:, k]] for k in range(s["positions"]))
    np.testing.assert_allclose(out["emb_sum"], want, rtol=1e-14)


def test_draw_offset_is_base_plus_group():
    """Group j of row r draws from its own logits with Philox row index r, the
    row's seed and offset[r] + j."""
    from oracle.draw import draw
    s, w, h, c0, sp = _tiny(rows=2, kind="fixed")
    a = run_frame(s, w, h, c0, sp, "fp64")
    for r in range(2):
        for j in range(s["positions"] - 1):
            lg = a["logits"][j, r].astype(np.float32)
            assert a["drawn"][r, j] == draw(lg, 0.9, 50, 0.8, r, r, j)


# ---------------------------------------------------------------- library check
def _torch_sequence_frame(s, w, h, codes):
    """The same frame written the other way round: with the codes fixed, the
    depth loop is one causal pass of the transformer over the whole sequence
    [in_proj(h), E_0(c_0), ..., E_{P-2}(c_{P-2})], built from torch's functional
    ops (rms_norm, linear, scaled_dot_product_attention with GQA, silu) in fp64."""
    F = torch.nn.functional
    T = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))  # noqa: E731
    W = {k: T(synth.bf16_bits_to_f32(v)) for k, v in w.items()}
    L, H, Hq, Hkv, D, P = (s["layers"], s["hidden"], s["q_heads"], s["kv_heads"],
                           s["head_dim"], s["positions"])
    eps, base = s["rms_eps"], s["rope_base"]
    R = h.shape[0]
    seq = [F.linear(T(h), W["in_proj"])]
    for j in range(P - 1):
        seq.append(W["embed"][j][torch.from_numpy(codes[:, j].astype(np.int64))])
    x = torch.stack(seq, dim=1)                                   # [R][P][H]
    inv = base ** (-2.0 * torch.arange(D // 2, dtype=torch.float64) / D)
    ang = torch.arange(P, dtype=torch.float64)[:, None] * inv[None, :]
    cos, sin = torch.cos(ang), torch.sin(ang)

    def rot(t):                                                   # [R][heads][P][D]
        a, b = t[..., :D // 2], t[..., D // 2:]
        return torch.cat([a * cos - b * sin, b * cos + a * sin], dim=-1)

    for l in range(L):
        a = F.rms_norm(x, (H,), W["attn_norm"][l], eps=eps)
        qkv = F.linear(a, W["w_qkv"][l])
        q = qkv[..., :Hq * D].reshape(R, P, Hq, D)
        k = qkv[..., Hq * D:(Hq + Hkv) * D].reshape(R, P, Hkv, D)
        v = qkv[..., (Hq + Hkv) * D:].reshape(R, P, Hkv, D)
        q = F.rms_norm(q, (D,), W["q_norm"][l], eps=eps).transpose(1, 2)
        k = F.rms_norm(k, (D,), W["k_norm"][l], eps=eps).transpose(1, 2)
        o = F.scaled_dot_product_attention(rot(q), rot(k), v.transpose(1, 2),
                                           is_causal=True, enable_gqa=True)
        x = x + F.linear(o.transpose(1, 2).reshape(R, P, Hq * D), W["w_o"][l])
        a = F.rms_norm(x, (H,), W["mlp_norm"][l], eps=eps)
        x = x + F.linear(F.silu(F.linear(a, W["w_gate"][l])) * F.linear(a, W["w_up"][l]),
                         W["w_down"][l])
    y = F.rms_norm(x, (H,), W["final_norm"], eps=eps)
    return torch.stack([F.linear(y[:, j + 1], W["heads"][j]) for j in range(P - 1)]).numpy()


@pytest.mark.parametrize("kind", ["greedy", "mixed"])
def test_frame_matches_torch_full_sequence_pass(kind):
    s, w, h, c0, sp = _tiny(rows=3, kind=kind, seed=4)
    out = run_frame(s, w, h, c0, sp, "fp64")
    codes = np.concatenate([c0[:, None], out["codes"]], axis=1)
    want = _torch_sequence_frame(s, w, h, codes)
    np.testing.assert_allclose(out["logits"], want, rtol=1e-10, atol=1e-12)


def test_bf16_operands_stay_within_the_logit_tolerance_of_fp64():
    s, w, h, c0, sp = _tiny(rows=4)
    a = run_frame(s, w, h, c0, sp, "fp64")
    b = run_frame(s, w, h, c0, sp, "bf16io", forced_codes=a["codes"])
    d = a["logits"] - b["logits"]
    assert np.abs(d).max() <= 3e-2
    assert np.linalg.norm(d) / np.linalg.norm(a["logits"]) <= 1e-2
    assert 0 < np.abs(d).max()          # the rounding points are really applied


# ---------------------------------------------------------------- bf16 operand of a norm
def test_bf16_operand_of_a_norm_is_its_output_rounded_once():
    """Where the bf16-operand mode rounds the input of a normed projection,
    pinned on a hand-worked case in which the plausible placements disagree.

    y = [1, 2, 3, 5], gain = [1.5, 0.75, 1.25, 1.0625], eps = 0:
    mean(y^2) = 39/4, so the row factor r = (39/4)^(-1/2) = 0.32025630761...
    and the norm's output y * r * gain = [0.480384461, 0.480384461,
    1.200961154, 1.701361634]. bf16 keeps 8 significant bits: the ulp is 2^-9
    on [0.25, 0.5) and 2^-7 on [1, 2), so the nearest values are 246 * 2^-9,
    246 * 2^-9, 154 * 2^-7 and 218 * 2^-7 (bit patterns 3ef6 3ef6 3f9a 3fda).
    The other placement (round y * gain, then scale the product by r) rounds
    nothing here: y * gain = [1.5, 1.5, 3.75, 5.3125] is exact in bf16, so a
    projection onto a row of ones would give 12.0625 * r = 3.863091710...,
    while the norm's rounded output gives 3.8671875."""
    from oracle.frame import norm_operand
    y = np.array([[1.0, 2.0, 3.0, 5.0]])
    g = np.array([1.5, 0.75, 1.25, 1.0625])
    got = norm_operand(y, g, 0.0, "bf16io")
    np.testing.assert_array_equal(got[0], [0.48046875, 0.48046875, 1.203125, 1.703125])
    bits = got.astype(np.float32).view(np.uint32)[0] >> 16
    assert [int(b) for b in bits] == [0x3EF6, 0x3EF6, 0x3F9A, 0x3FDA]
    assert float(got[0] @ np.ones(4)) == 3.8671875
    exact = norm_operand(y, g, 0.0, "fp64")
    assert abs(float(exact[0] @ np.ones(4)) - 12.0625 / np.sqrt(39 / 4)) < 1e-15
    assert abs(12.0625 / np.sqrt(39 / 4) - 3.863091710547727) < 1e-15


def test_frame_projects_the_rounded_norm_output(monkeypatch):
    """The frame's normed projections (qkv, gate/up, heads) read their operand
    through norm_operand: swapping in the other placement (y * gain rounded,
    the row factor applied to the product) changes the bf16-operand logits,
    and leaves the float64 ones untouched."""
    import oracle.frame as fr
    s, w, h, c0, sp = _tiny(rows=2)
    a16 = run_frame(s, w, h, c0, sp, "bf16io")
    a64 = run_frame(s, w, h, c0, sp, "fp64")

    def other(y, gain, eps, mode):
        if mode != "bf16io":
            return fr.rms_norm(y, gain, eps)
        f = 1.0 / np.sqrt(np.mean(y * y, axis=-1, keepdims=True) + eps)
        return fr.bf16_round(y * gain) * f

    monkeypatch.setattr(fr, "norm_operand", other)
    b16 = run_frame(s, w, h, c0, sp, "bf16io", forced_codes=a16["codes"])
    b64 = run_frame(s, w, h, c0, sp, "fp64", forced_codes=a64["codes"])
    np.testing.assert_array_equal(a64["logits"], b64["logits"])
    assert np.abs(a16["logits"] - b16["logits"]).max() > 0
