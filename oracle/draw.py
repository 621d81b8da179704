"""The per-row draw: temperature, top-k, top-p, then Gumbel-max on Philox uniforms.

Test infrastructure only (see oracle/__init__.py).

"Qwen3-TTS: Run the 1.7B Depth Loop as One Persistent Kernel on Hopper",
section "How it works": a draw reads the row's temperature, top-k, top-p, seed
and offset and picks one token, as one plain sample call would. The pages give
no formula for the filters; the reading taken here (the common serving order):

1. temperature <= 0: the token with the largest logit, ties to the lowest index.
2. otherwise s = logit / temperature (float32).
3. top-k with 1 <= k < vocab: keep the k tokens that come first in the order
   (s descending, index ascending); k = 0 or k >= vocab keeps every token.
4. top-p < 1: softmax over the kept tokens, walk them in the same order and
   keep a token while the probability mass of the tokens before it is below p
   (the first token is always kept).
5. Gumbel-max: u_v from Philox4x32-10 (oracle.philox), the token maximising
   s_v - log(-log u_v) over the kept set, ties to the lowest index.

The draw decides an integer from floating point, so it runs in float32, the
precision of the CUDA kernel.
"""
from __future__ import annotations

import numpy as np

from .philox import vocab_uniforms

F32 = np.float32


def _order(s: np.ndarray) -> np.ndarray:
    """Indices sorted by (s descending, index ascending)."""
    idx = np.arange(s.shape[0])
    return np.lexsort((idx, -s))


def draw_detail(logits, temperature, top_k, top_p, seed, row, offset) -> dict:
    """One draw with the quantities its decision turns on.

    Returns ``code`` plus, for judging near-ties between two implementations:
    ``margin`` -- gap between the best and second-best score that decided the
    code, in logit units (logit gap when greedy; perturbed-score gap times the
    temperature otherwise; inf when only one candidate);
    ``topk_gap`` -- gap between the k-th and (k+1)-th logit (inf when top-k is off);
    ``topp_gap`` -- smallest |mass-before - p| over the top-k tokens (inf when off).
    """
    lg = np.asarray(logits, dtype=F32)
    V = lg.shape[0]
    T = F32(temperature)
    inf = float("inf")
    if not (T > 0):
        best = lg.max()
        code = int(np.flatnonzero(lg == best).min())
        rest = np.delete(lg, code)
        margin = float(best - rest.max()) if rest.size else inf
        return dict(code=code, margin=margin, topk_gap=inf, topp_gap=inf)

    s = (lg / T).astype(F32)
    order = _order(s)
    k = int(top_k)
    kept = order
    topk_gap = inf
    if 1 <= k < V:
        kept = order[:k]
        topk_gap = float((s[order[k - 1]] - s[order[k]]) * T)
    p = F32(top_p)
    topp_gap = inf
    if p < 1:
        sk = s[kept]
        e = np.exp((sk - sk[0]).astype(F32)).astype(F32)
        z = F32(np.cumsum(e, dtype=F32)[-1])
        prob = (e / z).astype(F32)
        before = np.concatenate([[F32(0)], np.cumsum(prob, dtype=F32)[:-1]]).astype(F32)
        keep = before < p
        keep[0] = True
        topp_gap = float(np.abs(before.astype(np.float64) - float(p)).min())
        kept = kept[keep]

    u = vocab_uniforms(seed, row, offset, V)
    g = (-np.log(-np.log(u))).astype(F32)
    zv = (s[kept] + g[kept]).astype(F32)
    best = zv.max()
    code = int(kept[zv == best].min())
    others = zv[kept != code]
    margin = float((best - others.max()) * T) if others.size else inf
    return dict(code=code, margin=margin, topk_gap=topk_gap, topp_gap=topp_gap)


def draw(logits, temperature, top_k, top_p, seed, row, offset) -> int:
    """The token one draw picks (see the module docstring)."""
    return draw_detail(logits, temperature, top_k, top_p, seed, row, offset)["code"]
