"""Consumer of the decompressed gradient: global-norm clipping and an Adam step, in fp64.

TEST INFRASTRUCTURE, like the rest of this package: only ``tests/`` may import it. It
shares no code with the CUDA path.

Sources:
  [card] "Zero-Shot Text-to-Image Generation - 中文验证版", §方法适配: the training used
         Adam, with gradient clipping and a skip-update rule for nonfinite values. The
         moments' custom 16-bit format is not specified there, so the moments here are
         fp32 state.
  [amp]  "AIGC 基本功|混合精度与数值稳定性", §6.2 and its clipping paragraph: the norm
         used for clipping is global, the square root of the sum of every shard's local
         sum of squares. Clipping comes after unscaling and the nonfinite check, and the
         order is: unscale, check nonfinite, global norm, clip, optimizer step, update
         the scale. A skipped step updates nothing.

The Adam update itself is the published algorithm (Kingma and Ba, 2015) with bias
correction, restated plainly:
  m <- b1 m + (1 - b1) g;  v <- b2 v + (1 - b2) g^2
  theta <- theta - lr * (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps)
Clipping is the usual global rescale g <- g * min(1, C / ||g||); a zero norm leaves g
unchanged. The pages give neither an epsilon inside the ratio nor weight decay, so
there is none.

Parity status: global_norm, clip_coefficient and adam_step are pinned in
tests/test_oracle_pins.py. global_norm is checked against a norm computed over the
concatenation of the shards. adam_step is checked against the closed forms of its first
step (lr * g / (|g| + eps)) and of a constant gradient (the step tends to lr), and by
its invariance to a positive rescaling of the gradient when eps = 0. clip_coefficient
is checked by hand-worked values.
"""
from __future__ import annotations

import math

import numpy as np


def global_norm(shards) -> float:
    """||g||_2 over every shard: sqrt(sum over shards of the local sum of squares), fp64.
    [amp] §6.2: each shard contributes its local sum of squares, and the sums are
    all-reduced before the root."""
    total = 0.0
    for s in shards:
        a = np.asarray(s, dtype=np.float64)
        total += float(np.sum(a * a))
    return math.sqrt(total)


def clip_coefficient(norm: float, max_norm: float) -> float:
    """min(1, C / ||g||); 1 when ||g|| = 0 (nothing to clip)."""
    if norm <= max_norm or norm == 0.0:
        return 1.0
    return float(max_norm) / float(norm)


def adam_step(theta, m, v, g, t: int, lr: float, beta1: float, beta2: float, eps: float,
              clip: float = 1.0, skip: bool = False):
    """One Adam step on fp64 copies of the fp32 state (theta, m, v), t >= 1 the step
    number after this update, g the (unclipped) gradient and `clip` its clip
    coefficient. A skipped step returns the state unchanged. Returns (theta, m, v)."""
    theta = np.asarray(theta, dtype=np.float64)
    m = np.asarray(m, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if skip:
        return theta.copy(), m.copy(), v.copy()
    gc = np.asarray(g, dtype=np.float64) * float(clip)
    m_new = beta1 * m + (1.0 - beta1) * gc
    v_new = beta2 * v + (1.0 - beta2) * gc * gc
    m_hat = m_new / (1.0 - beta1 ** t)
    v_hat = v_new / (1.0 - beta2 ** t)
    theta_new = theta - lr * m_hat / (np.sqrt(v_hat) + eps)
    return theta_new, m_new, v_new
