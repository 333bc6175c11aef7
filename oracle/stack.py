"""fp64 oracle for the layer-streaming stack: L decoder layers, lm-head
cross-entropy, backward in reverse, global gradient-norm clipping.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources: "From-scratch GPU LLM training", capability list (layer-streaming
forward holding one layer at a time, lossless against the bulk forward; the
end-to-end smoke bullet trains under gradient clipping). Streaming changes
where weights live, never the arithmetic, so the oracle runs the stack in
bulk.

Readings: the hidden states of the last layer feed the lm-head directly (no
final norm); the global norm covers every weight gradient (7 projections and
2 gains per layer, plus the lm-head weight), not dX; the clip coefficient is
min(1, max_norm / (norm + 1e-6)) and multiplies every weight gradient.
"""
from __future__ import annotations

import numpy as np

from .qwen3_layer import LayerConfig, layer_backward, layer_forward, lmhead_ce

CLIP_EPS = 1e-6


def clip_coefficient(total_norm: float, max_norm: float) -> float:
    return min(1.0, max_norm / (total_norm + CLIP_EPS))


def stack_fwd_bwd(cfg: LayerConfig, layers: list, W_lm: np.ndarray, X: np.ndarray,
                  targets: np.ndarray, max_norm: float):
    """Returns dict(loss, argmax, total_norm, clip_coef, grads (list per layer,
    clipped), dW_lm (clipped), dX (unclipped input gradient), Y_last)."""
    x = np.asarray(X, np.float64)
    saved = []
    for w in layers:
        x, s = layer_forward(cfg, w, x)
        saved.append(s)
    head = lmhead_ce(x, W_lm, targets)
    dx = head["dX"]
    grads = [None] * len(layers)
    for li in range(len(layers) - 1, -1, -1):
        dx, g, _ = layer_backward(cfg, layers[li], saved[li], dx)
        grads[li] = g
    sq = float(np.sum(head["dW"] ** 2))
    for g in grads:
        for name in g:
            sq += float(np.sum(g[name] ** 2))
    total_norm = float(np.sqrt(sq))
    coef = clip_coefficient(total_norm, max_norm)
    grads = [{k: v * coef for k, v in g.items()} for g in grads]
    return dict(loss=head["loss"], argmax=head["argmax"], total_norm=total_norm,
                clip_coef=coef, grads=grads, dW_lm=head["dW"] * coef, dX=dx,
                Y_last=x)
