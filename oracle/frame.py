"""One frame of the codec-TTS depth decoder, written out plainly in float64.

Test infrastructure only (see oracle/__init__.py).

What a frame computes ("Qwen3-TTS: Run the 1.7B Depth Loop as One Persistent
Kernel on Hopper", sections "How it works" and "What's left in the frame,
open"): a 5-layer CodePredictor stepped over 16 depth positions; an input
projection; 16 embedding steps, 15 of which first draw a code from one of 15
heads. The transformer layer is the Qwen3 layer named in "The gaps between
kernels: PDL and megakernels", section "How large are the gaps: an estimate"
(RMSNorm before attention and before the MLP, QK-Norm plus RoPE, a SwiGLU MLP,
residual adds), with grouped-query attention (section "How it works" of the
first page: an attention task waits on the qkv tiles of its kv head).

Readings taken where the pages are silent:
* position 0's input is the input projection of the talker hidden state;
  position 1's input is table 0's embedding of the first code; head j reads
  position j+1's output and its code j+1 is embedded by table j+1 as position
  j+2's input (the last only feeds the embedding sum);
* one shared final RMSNorm before every head; no biases;
* QK-Norm is a per-head RMSNorm over head_dim with its own gain; RoPE is the
  rotate-half form on pairs (i, i + D/2) with angle pos * base^(-2i/D),
  positions 0..P-1 inside the frame;
* q head h reads kv head floor(h / (Hq / Hkv));
* every draw advances nothing inside the frame; group j of row r draws at
  offset[r] + j and the frame returns offset[r] + P - 1 for every row.

Two precisions:
* ``"fp64"``: nothing is rounded; the reference for the logit tolerance.
* ``"bf16io"``: values are rounded to bfloat16 exactly where they become the
  operand of a bf16 projection tile or of attention: the talker hidden state,
  each RMSNorm's output x * (mean(x^2) + eps)^(-1/2) * gain (rounded once,
  after the gain), q/k/v after QK-Norm and RoPE, the attention output,
  silu(gate) * up. Everything else stays float64. The pages make every
  projection a bf16 tile (section "How it works") of the Qwen3 layer, where a
  projection after a norm reads that norm's output: so the value rounded to
  bf16 is the norm's output itself, gain included.
"""
from __future__ import annotations

import numpy as np

from .draw import draw_detail

F64 = np.float64


def bf16_round(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value (ties to even).

    bfloat16 keeps 8 significant bits; the float64 significand has 53, so 45
    low bits are dropped with round-to-nearest-even on the bit pattern. Valid
    for values in the normal range of float32 (all values here)."""
    a = np.ascontiguousarray(x, dtype=F64)
    b = a.view(np.uint64)
    lsb = (b >> np.uint64(45)) & np.uint64(1)
    r = (b + np.uint64((1 << 44) - 1) + lsb) & ~np.uint64((1 << 45) - 1)
    return r.view(F64)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """The values encoded by bfloat16 bit patterns (uint16)."""
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(F64)


def rms_norm(v, gain, eps) -> np.ndarray:
    """v * (mean(v^2) + eps)^(-1/2) * gain over the last axis."""
    v = np.asarray(v, dtype=F64)
    return v / np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + eps) * gain


def rope(v, pos, base) -> np.ndarray:
    """Rotate-half RoPE at position ``pos`` over the last axis (length D):
    pair (i, i + D/2) turns by angle pos * base^(-2i/D)."""
    v = np.asarray(v, dtype=F64)
    D = v.shape[-1]
    half = D // 2
    ang = pos * base ** (-2.0 * np.arange(half, dtype=F64) / D)
    c, s = np.cos(ang), np.sin(ang)
    a, b = v[..., :half], v[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def norm_operand(y, gain, eps, mode: str) -> np.ndarray:
    """The bf16 projection operand that an RMSNorm feeds: rms_norm(y, gain),
    rounded to bfloat16 once in ``"bf16io"`` mode ("Qwen3-TTS: Run the 1.7B
    Depth Loop as One Persistent Kernel on Hopper", section "How it works":
    the projections are bf16 tiles; the norm precedes qkv, gate/up and the
    heads as in the Qwen3 layer)."""
    a = rms_norm(y, gain, eps)
    return bf16_round(a) if mode == "bf16io" else a


def silu(z) -> np.ndarray:
    """z / (1 + exp(-z))."""
    z = np.asarray(z, dtype=F64)
    return z / (1.0 + np.exp(-z))


def attention(q, K, V) -> np.ndarray:
    """Causal attention of one position over the frame's positions so far.

    q: [R][Hq][D] at the current position; K, V: [T][R][Hkv][D] for positions
    0..T-1 (the current one last). q head h reads kv head h // (Hq / Hkv).
    Returns [R][Hq][D] = sum_t softmax_t(q . k_t / sqrt(D)) v_t."""
    R, Hq, D = q.shape
    Hkv = K.shape[2]
    grp = Hq // Hkv
    kv_of = np.arange(Hq) // grp
    Kh = K[:, :, kv_of, :]                          # [T][R][Hq][D]
    Vh = V[:, :, kv_of, :]
    sc = np.einsum("rhd,trhd->rht", q, Kh) / np.sqrt(D)
    sc = sc - sc.max(axis=-1, keepdims=True)
    w = np.exp(sc)
    w = w / w.sum(axis=-1, keepdims=True)
    return np.einsum("rht,trhd->rhd", w, Vh)


class Weights:
    """float64 views of the bf16 weights (converted once, on first use)."""

    def __init__(self, bits: dict):
        self.bits = bits
        self._cache = {}

    def __getitem__(self, name):
        if name not in self._cache:
            self._cache[name] = bf16_bits_to_f64(self.bits[name])
        return self._cache[name]


def run_frame(shape: dict, weights, h, first_code, sampler: dict, mode: str = "fp64",
              forced_codes=None, keep_kv: bool = False) -> dict:
    """Run one frame for all rows.

    ``weights``: dict of bf16 bit arrays (synth.weights layout) or a Weights.
    ``h``: float32 [R][T_h]; ``first_code``: int [R]; ``sampler``: dict of
    per-row arrays temperature, top_k, top_p, seed, offset.
    ``forced_codes``: optional int [R][P-1]; when given, those codes are
    embedded instead of the drawn ones (teacher forcing) and ``drawn`` still
    reports what this oracle would draw at each forced prefix.

    Returns dict with ``codes`` [R][P-1] (the codes embedded), ``drawn``
    [R][P-1], ``detail`` (per row and group, see oracle.draw.draw_detail),
    ``logits`` [P-1][R][V] float64, ``emb_sum`` [R][H], ``offset`` [R] and,
    with ``keep_kv``, ``K``/``V`` [L][P][R][Hkv][D] and ``x_out`` [P][R][H]
    (each position's output).
    """
    if mode not in ("fp64", "bf16io"):
        raise ValueError(mode)
    W = weights if isinstance(weights, Weights) else Weights(weights)
    rnd = bf16_round if mode == "bf16io" else (lambda a: np.asarray(a, dtype=F64))
    L, H, Hq, Hkv, D = (shape["layers"], shape["hidden"], shape["q_heads"],
                        shape["kv_heads"], shape["head_dim"])
    P, V = shape["positions"], shape["vocab"]
    eps, base, qkn = float(shape["rms_eps"]), float(shape["rope_base"]), bool(shape["qk_norm"])
    h = np.asarray(h, dtype=np.float32)
    R = h.shape[0]
    c0 = np.asarray(first_code, dtype=np.int64)

    x_in = [None] * (P + 1)
    x_in[0] = rnd(h.astype(F64)) @ W["in_proj"].T
    x_in[1] = W["embed"][0][c0].copy()
    emb_sum = W["embed"][0][c0].copy()

    Kc = np.zeros((L, P, R, Hkv, D))
    Vc = np.zeros((L, P, R, Hkv, D))
    codes = np.zeros((R, P - 1), dtype=np.int32)
    drawn = np.zeros((R, P - 1), dtype=np.int32)
    logits = np.zeros((P - 1, R, V))
    detail = [[None] * (P - 1) for _ in range(R)]
    x_out = np.zeros((P, R, H))

    def normed(y, gain, wt):
        """The projection of the norm's output (rounded once to bf16 in
        bf16io mode: it is the tile's operand)."""
        return norm_operand(y, gain, eps, mode) @ wt

    for p in range(P):
        y = x_in[p].copy()
        for l in range(L):
            qkv = normed(y, W["attn_norm"][l], W["w_qkv"][l].T)
            q = qkv[:, :Hq * D].reshape(R, Hq, D)
            k = qkv[:, Hq * D:(Hq + Hkv) * D].reshape(R, Hkv, D)
            v = qkv[:, (Hq + Hkv) * D:].reshape(R, Hkv, D)
            if qkn:
                q = rms_norm(q, W["q_norm"][l], eps)
                k = rms_norm(k, W["k_norm"][l], eps)
            Kc[l, p] = rnd(rope(k, p, base))
            Vc[l, p] = rnd(v)
            o = attention(rnd(rope(q, p, base)), Kc[l, :p + 1], Vc[l, :p + 1])
            y = y + rnd(o.reshape(R, Hq * D)) @ W["w_o"][l].T
            m = rnd(silu(normed(y, W["mlp_norm"][l], W["w_gate"][l].T))
                    * normed(y, W["mlp_norm"][l], W["w_up"][l].T))
            y = y + m @ W["w_down"][l].T
        x_out[p] = y
        if p >= 1:
            j = p - 1
            lg = normed(y, W["final_norm"], W["heads"][j].T)
            logits[j] = lg
            for r in range(R):
                d = draw_detail(lg[r].astype(np.float32), sampler["temperature"][r],
                                sampler["top_k"][r], sampler["top_p"][r],
                                int(sampler["seed"][r]), r, int(sampler["offset"][r]) + j)
                detail[r][j] = d
                drawn[r, j] = d["code"]
            codes[:, j] = drawn[:, j] if forced_codes is None else np.asarray(forced_codes)[:, j]
            e = W["embed"][j + 1][codes[:, j].astype(np.int64)]
            x_in[p + 1] = e
            emb_sum = emb_sum + e

    out = dict(codes=codes, drawn=drawn, detail=detail, logits=logits, emb_sum=emb_sum,
               offset=np.asarray(sampler["offset"], dtype=np.int64) + (P - 1))
    if keep_kv:
        out.update(K=Kc, V=Vc, x_out=x_out)
    return out
