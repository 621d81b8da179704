"""Seeded synthetic inputs for the depth-decoder frame.

This module is the only code shared by the CPU oracle and the CUDA path. It
holds no arithmetic of the method itself: it draws weights, talker hidden
states, first codes and per-row sampler settings from seeded generators and
hands them out as plain numpy arrays.

Recipe (the shapes are those of the workloads quoted for the Qwen3-TTS 1.7B
CodePredictor depth loop; the distributions stand in for the real checkpoint,
which is not available):

* every weight matrix, embedding table and head: N(0, 0.02), drawn in float32
  and rounded to bfloat16 (round to nearest even, done by torch's dtype cast);
* every norm gain (attention, MLP, final, per-head q/k norms): 1 + N(0, 0.01),
  rounded to bfloat16 the same way;
* talker hidden state: float32 N(0, 1);
* first code: uniform integer in [0, vocab);
* sampler settings: see :func:`sampler`.

Each tensor gets its own stream: numpy's PCG64 seeded from
``SeedSequence(master_seed, spawn_key=(tensor_id,))``, so a tensor does not
depend on the order in which others are drawn. Per-row Philox seeds in the
mixed sampler come from SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) over the row index.
"""
from __future__ import annotations

import numpy as np

__all__ = ["SHAPES", "shape", "weights", "talker_hidden", "first_codes",
           "sampler", "splitmix64", "bf16_bits_to_f32", "weight_bytes_per_frame"]

# Shapes. Field names follow the C header's cp_shape.
SHAPES = {
    # 1 layer, hidden 256, 4 q / 2 kv heads of 64, FFN 768, 4 depth positions,
    # 3 heads of vocab 256, input projection 512 -> 256.
    "tiny": dict(layers=1, hidden=256, q_heads=4, kv_heads=2, head_dim=64, ffn=768,
                 positions=4, vocab=256, talker_hidden=512, max_rows=64,
                 rms_eps=1e-6, rope_base=10000.0, qk_norm=1),
    # The 1.7B CodePredictor: 5 layers, hidden 1024, 16 q / 8 kv heads of 128,
    # FFN 3072, 16 depth positions, 15 heads and 16 tables of vocab 2048,
    # input projection 2048 -> 1024.
    "full": dict(layers=5, hidden=1024, q_heads=16, kv_heads=8, head_dim=128, ffn=3072,
                 positions=16, vocab=2048, talker_hidden=2048, max_rows=64,
                 rms_eps=1e-6, rope_base=10000.0, qk_norm=1),
    # Twice as wide: hidden 2048, 16 q / 16 kv heads of 128, FFN 6144.
    "wide": dict(layers=5, hidden=2048, q_heads=16, kv_heads=16, head_dim=128, ffn=6144,
                 positions=16, vocab=2048, talker_hidden=2048, max_rows=64,
                 rms_eps=1e-6, rope_base=10000.0, qk_norm=1),
}
# The same decoders with room for 128 rows a frame (M = 128 projections).
SHAPES["full_r128"] = dict(SHAPES["full"], max_rows=128)
SHAPES["tiny_r128"] = dict(SHAPES["tiny"], max_rows=128)

_TENSOR_IDS = {
    "in_proj": 1, "embed": 2, "attn_norm": 3, "mlp_norm": 4, "q_norm": 5, "k_norm": 6,
    "w_qkv": 7, "w_o": 8, "w_gate": 9, "w_up": 10, "w_down": 11, "final_norm": 12,
    "heads": 13, "talker_hidden": 20, "first_codes": 21, "sampler": 22,
}


def shape(name: str) -> dict:
    """A copy of one of the named shapes."""
    return dict(SHAPES[name])


def _rng(master: int, name: str) -> np.random.Generator:
    ss = np.random.SeedSequence(int(master), spawn_key=(_TENSOR_IDS[name],))
    return np.random.Generator(np.random.PCG64(ss))


def _to_bf16_bits(a: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns (uint16) to the float32 values they encode."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(master: int, name: str, shp, std: float, mean: float = 0.0) -> np.ndarray:
    g = _rng(master, name)
    a = g.standard_normal(size=shp, dtype=np.float32)
    a *= np.float32(std)
    if mean:
        a += np.float32(mean)
    return _to_bf16_bits(a)


def weights(s: dict, seed: int = 0) -> dict:
    """All weights of a frame as bfloat16 bit patterns (numpy uint16).

    Layouts are row-major ``[out][in]`` (the nn.Linear layout):
    in_proj [H][T_h]; embed [P][V][H]; attn_norm, mlp_norm [L][H];
    q_norm, k_norm [L][D]; w_qkv [L][(Hq+2Hkv)*D][H] with rows q | k | v;
    w_o [L][H][Hq*D]; w_gate, w_up [L][F][H]; w_down [L][H][F];
    final_norm [H]; heads [P-1][V][H].
    """
    L, H, Hq, Hkv, D, F = (s["layers"], s["hidden"], s["q_heads"], s["kv_heads"],
                           s["head_dim"], s["ffn"])
    P, V, T = s["positions"], s["vocab"], s["talker_hidden"]
    w = {}
    w["in_proj"] = _normal_bf16(seed, "in_proj", (H, T), 0.02)
    w["embed"] = _normal_bf16(seed, "embed", (P, V, H), 0.02)
    w["attn_norm"] = _normal_bf16(seed, "attn_norm", (L, H), 0.01, 1.0)
    w["mlp_norm"] = _normal_bf16(seed, "mlp_norm", (L, H), 0.01, 1.0)
    w["q_norm"] = _normal_bf16(seed, "q_norm", (L, D), 0.01, 1.0)
    w["k_norm"] = _normal_bf16(seed, "k_norm", (L, D), 0.01, 1.0)
    w["w_qkv"] = _normal_bf16(seed, "w_qkv", (L, (Hq + 2 * Hkv) * D, H), 0.02)
    w["w_o"] = _normal_bf16(seed, "w_o", (L, H, Hq * D), 0.02)
    w["w_gate"] = _normal_bf16(seed, "w_gate", (L, F, H), 0.02)
    w["w_up"] = _normal_bf16(seed, "w_up", (L, F, H), 0.02)
    w["w_down"] = _normal_bf16(seed, "w_down", (L, H, F), 0.02)
    w["final_norm"] = _normal_bf16(seed, "final_norm", (H,), 0.01, 1.0)
    w["heads"] = _normal_bf16(seed, "heads", (P - 1, V, H), 0.02)
    return w


def weight_bytes_per_frame(s: dict) -> int:
    """Bytes of weight matrices one frame streams: every layer once per depth
    position, each head once, the input projection once (embedding rows and
    norm gains are not counted)."""
    L, H, Hq, Hkv, D, F = (s["layers"], s["hidden"], s["q_heads"], s["kv_heads"],
                           s["head_dim"], s["ffn"])
    P, V, T = s["positions"], s["vocab"], s["talker_hidden"]
    per_layer = ((Hq + 2 * Hkv) * D * H + H * Hq * D + 2 * F * H + H * F) * 2
    return P * L * per_layer + (P - 1) * V * H * 2 + H * T * 2


def talker_hidden(s: dict, rows: int, seed: int = 0, frame: int = 0) -> np.ndarray:
    """float32 [rows][T_h] ~ N(0, 1). ``frame`` selects a fresh draw per frame."""
    ss = np.random.SeedSequence(int(seed), spawn_key=(_TENSOR_IDS["talker_hidden"], int(frame)))
    g = np.random.Generator(np.random.PCG64(ss))
    return g.standard_normal(size=(rows, s["talker_hidden"]), dtype=np.float32)


def first_codes(s: dict, rows: int, seed: int = 0) -> np.ndarray:
    """int32 [rows], uniform in [0, vocab)."""
    g = _rng(seed, "first_codes")
    return g.integers(0, s["vocab"], size=rows, dtype=np.int64).astype(np.int32)


_MASK64 = (1 << 64) - 1


def splitmix64(master: int, index: int) -> int:
    """SplitMix64 output number ``index`` of the stream started at ``master``."""
    z = (int(master) + (int(index) + 1) * 0x9E3779B97F4A7C15) & _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def sampler(kind: str, rows: int, seed: int = 0) -> dict:
    """Per-row sampler settings.

    ``greedy``: temperature 0 for every row.
    ``fixed``: temperature 0.9, top-k 50, top-p 0.8, Philox seed = row index,
    offset 0 (the 64-row sampled workload).
    ``mixed``: temperature U[0, 1.2], top-k from {0, 20, 50, 200}, top-p
    U[0.5, 1.0], Philox seed SplitMix64(master, row), offset 0 (the row sweep).
    """
    r = np.arange(rows)
    if kind == "greedy":
        out = dict(temperature=np.zeros(rows, np.float32), top_k=np.zeros(rows, np.int32),
                   top_p=np.ones(rows, np.float32), seed=r.astype(np.uint64),
                   offset=np.zeros(rows, np.int64))
    elif kind == "fixed":
        out = dict(temperature=np.full(rows, 0.9, np.float32), top_k=np.full(rows, 50, np.int32),
                   top_p=np.full(rows, 0.8, np.float32), seed=r.astype(np.uint64),
                   offset=np.zeros(rows, np.int64))
    elif kind == "mixed":
        g = _rng(seed, "sampler")
        out = dict(temperature=g.uniform(0.0, 1.2, size=rows).astype(np.float32),
                   top_k=np.array([0, 20, 50, 200], np.int32)[g.integers(0, 4, size=rows)],
                   top_p=g.uniform(0.5, 1.0, size=rows).astype(np.float32),
                   seed=np.array([splitmix64(seed, i) for i in r], dtype=np.uint64),
                   offset=np.zeros(rows, np.int64))
    else:
        raise ValueError(f"unknown sampler kind {kind!r}")
    return out
