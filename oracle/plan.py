"""The frame's phase sequence and its weight traffic, in closed form.

Test infrastructure only (see oracle/__init__.py).

"Qwen3-TTS: Run the 1.7B Depth Loop as One Persistent Kernel on Hopper",
section "How it works": a frame is qkv, attention, o, gate/up and down for each
layer at each depth position, plus the input projection, 15 heads and 16
embedding steps, 15 of which draw a code first. Section "Where the depth
loop's time goes": each position reads the layers' weights again, and the
heads are read once each.

Order taken here (the only causal one): the input projection and table 0's
embedding of the first code, then for each position p the layers in order,
and after each position p >= 1 the head p-1 followed by its draw and the
embedding that feeds position p+1.
"""
from __future__ import annotations


def phases(shape: dict) -> list:
    """List of (kind, layer, position, group) in execution order."""
    L, P = shape["layers"], shape["positions"]
    out = [("INPROJ", -1, 0, -1), ("EMB0", -1, 1, 0)]
    for p in range(P):
        for l in range(L):
            for kind in ("QKV", "ATTN", "O", "GU", "DOWN"):
                out.append((kind, l, p, -1))
        if p >= 1:
            out.append(("HEAD", -1, p, p - 1))
            out.append(("DRAW", -1, p, p - 1))
    return out


def weight_bytes(shape: dict) -> dict:
    """bf16 weight bytes: per layer, per position (all layers), per frame."""
    L, H, Hq, Hkv, D, F = (shape["layers"], shape["hidden"], shape["q_heads"],
                           shape["kv_heads"], shape["head_dim"], shape["ffn"])
    P, V, T = shape["positions"], shape["vocab"], shape["talker_hidden"]
    qkv = (Hq + 2 * Hkv) * D * H * 2
    o = H * Hq * D * 2
    gu = 2 * F * H * 2
    down = H * F * 2
    layer = qkv + o + gu + down
    heads = (P - 1) * V * H * 2
    inproj = H * T * 2
    return dict(qkv=qkv, o=o, gu=gu, down=down, layer=layer, layers=L * layer,
                heads=heads, inproj=inproj, frame=P * L * layer + heads + inproj)
