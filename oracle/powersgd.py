"""The PowerSGD compression step with error feedback and per-resblock unscaling, in fp64.

TEST INFRASTRUCTURE. This is the oracle the CUDA library is checked against. Only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s ``cpu_baseline`` / reference
leg may import or execute it. It shares no code with the CUDA path. It is plain and
slow on purpose: one block, one matrix and one worker at a time, numpy fp64
arithmetic, and storage rounding only where the step stores into a 16-bit or fp32
buffer.

Sources:
  [card]  "Zero-Shot Text-to-Image Generation - 中文验证版" (ai-papers.xuzou.cn reading
          card), sections 瓶颈, 方法适配 and 证据.
  [notes] "[논문 정리] Zero-Shot Text-to-Image Generation" (only-wanna.tistory.com),
          sections "Mixed-Precision Training", "Data parallel" and the PowerSGD list
          under "All-Gather와 Reduce Scatter".
  [amp]   "AIGC 基本功|混合精度与数值稳定性" (jefxiong.cn), §3.1, §3.2, §6.2 and §6.8.

The pages name the method and what it compresses, but they do not list its arithmetic.
The step below is the plain one-step power iteration with error feedback: the
gradient is unscaled, cleaned of nonfinite values and added into the error buffer.
One warm-started subspace-iteration step then runs with a worker mean at each of the
two exchange points, and the error buffer keeps the residual. Where the pages leave
a detail open, the docstring says which reading is taken.

Parity status per function:
  unscale_and_mask, accumulate_error, skip_threshold, skip_block: pinned by brute force
    over all fp16 bit patterns and by the pages' printed fp16/bf16 values.
  power_step, error_update: pinned by a hand-worked 2x2 example, exact reconstruction
    of planted low rank, orthonormality, the linearity of the worker mean, basis
    invariance (Householder vs Gram-Schmidt), the error-feedback identity and the
    Eckart-Young bound.
  uncompressed_mean: pinned by a hand-worked example and the nonfinite brute force.
  scale_update: pinned by the closed form 2^(e0 + growths - backoffs) for power-of-two
    factors over a long random finite/nonfinite sequence, by hand-worked sequences that
    include a drop below 1, and by the fp32 product of a non-power-of-two factor.
  The values of P-hat and Q themselves depend on the basis and are not compared.
  Only G-hat, E, masks, counts and skips are compared.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from .numerics import round_to_format


# --------------------------------------------------------------------------- ingest
def unscale_and_mask(g_raw: np.ndarray, scale: float):
    """Unscale one resblock's gradient and zero its nonfinite entries.

    [notes] Mixed-Precision Training: each resblock scales its gradient when backprop
    enters the block and unscales it when the block ends. Inf/NaN values are set to 0
    there, because otherwise they cause underflow in other blocks. [card] 方法适配:
    every resblock has its own scale factor.

    Returns (g, mask). g = G_raw / s_b in fp64 with nonfinite entries set to 0, and
    mask = ~isfinite(G_raw / s_b). For the power-of-two scales the configurations use,
    the division is exact.
    """
    g = np.asarray(g_raw, dtype=np.float64) / float(scale)
    mask = ~np.isfinite(g)
    g = np.where(mask, 0.0, g)
    return g, mask


def accumulate_error(g: np.ndarray, e: np.ndarray, err_fmt: str) -> np.ndarray:
    """M = round_E(g + E): the cleaned gradient accumulated into the error buffer.

    [notes] PowerSGD list: the gradient is accumulated into the error buffer during
    backprop, which saves the memory of a separate buffer. Accumulating into the buffer
    means that M takes the buffer's storage type, so the fp64 sum is rounded once, RNE,
    to that type. The sum of two values of at most 24 significant bits is exact in fp64
    unless their exponents are far apart. In that case fp64's 53 bits still make the
    second rounding innocuous, since 53 >= 2p + 2 for every storage format used here.
    """
    return round_to_format(g + e, err_fmt)


def skip_threshold(fraction: float, workers: int, numel_block: int) -> int:
    """Integer count at or above which a block counts as nonfinite: ceil(T * W * numel).

    [card] 方法适配: the Adam update has a skip rule for nonfinite values. [amp] §6.2:
    every data-parallel rank must reach the same decision. Here the rule is a per-block
    integer threshold on the nonfinite count, summed over every worker and every
    gradient of the block. The threshold is computed in IEEE double from T.
    """
    return int(math.ceil(float(fraction) * float(workers * numel_block)))


def skip_block(counts_per_worker, threshold: int) -> bool:
    return int(np.sum(np.asarray(counts_per_worker, dtype=np.int64))) >= int(threshold)


def scale_update(scale: float, streak: int, counts_per_worker, backoff: float, growth: float,
                 interval: int):
    """One update of a resblock's dynamic gradient scale S and its finite-step streak.

    [amp] §3.2, the dynamic scaler: S becomes beta S when the scaled gradient holds an
    Inf or NaN, gamma S after K consecutive finite steps, and otherwise stays; beta < 1
    is the backoff, gamma > 1 the growth, K the interval. The page also notes that S is
    not guaranteed to stay above 1. [card] 方法适配 gives every resblock its own scale, so
    the rule runs per block. Here:
    - "holds an Inf or NaN" means the block's nonfinite count, summed over every worker,
      is > 0. That is the count the step reports, so every worker agrees ([amp] §6.2).
    - The streak counts consecutive finite steps. It restarts at 0 after a growth and
      after a backoff.
    - S is fp32 state. Each update is one IEEE single multiply by the factor rounded to
      fp32.
    - The page leaves open what happens when S leaves fp32's range. Here an update whose
      fp32 product is not a finite normal number (it overflows, or falls below 2^-126)
      keeps S, and the streak restarts as if the update had happened. A scale of 0 or
      Inf would turn every unscaled entry into a nonfinite value or into 0.

    Returns (S', streak').
    """
    s = np.float32(scale)

    def scaled(f):
        with np.errstate(over="ignore", under="ignore"):
            t = np.float32(s * np.float32(f))
        return t if (np.isfinite(t) and abs(float(t)) >= 2.0 ** -126) else s

    if int(np.sum(np.asarray(counts_per_worker, dtype=np.int64))) > 0:
        return scaled(backoff), 0
    streak = int(streak) + 1
    if streak >= int(interval):
        return scaled(growth), 0
    return s, streak


# ----------------------------------------------------------------------- power step
def orthonormalize(p: np.ndarray, method: str = "householder") -> np.ndarray:
    """Orthonormal basis of span(P), as many columns as P.

    The default is Householder QR (LAPACK through numpy). "mgs2" is modified
    Gram-Schmidt with one re-orthogonalisation pass, written out. It is kept so that a
    pin can show that the step does not depend on which orthonormal basis is chosen.
    """
    if method == "householder":
        qm, _ = np.linalg.qr(p, mode="reduced")
        return qm
    if method == "mgs2":
        v = np.array(p, dtype=np.float64, copy=True)
        m, r = v.shape
        for k in range(r):
            col = v[:, k].copy()
            for _ in range(2):
                for i in range(k):
                    col -= (v[:, i] @ col) * v[:, i]
            nrm = np.linalg.norm(col)
            v[:, k] = col / nrm if nrm > 0 else 0.0
        return v
    raise ValueError(method)


@dataclass
class PowerStepResult:
    p: np.ndarray  # mean of the per-worker P_w, m x r
    p_hat: np.ndarray  # orthonormal basis of span(P), m x r
    q: np.ndarray  # new Q (fp32 values held in fp64), n x r
    g_hat: np.ndarray  # decompressed gradient P_hat Q^T, m x n


def power_step(ms, q: np.ndarray, orth: str = "householder") -> PowerStepResult:
    """One warm-started subspace-iteration step over W workers that share Q.

    [card] 方法适配: the low-rank factors are all-reduced between machines instead of
    the full gradient. [notes] Data parallel: the workers' results are averaged. The
    steps, with Q (n x r) the persistent factor:
      P_w = M_w Q for every worker, then P = (1/W) sum_w P_w   (first exchange point)
      P_hat = an orthonormal basis of span(P)
      Q_w = M_w^T P_hat for every worker, then Q = (1/W) sum_w Q_w   (second exchange)
      Q is stored in fp32 (its state type)
      G_hat = P_hat Q^T   ([card] 证据: the decompressed gradient uses 32-bit products)
    Each worker's product is formed on its own, and only then averaged. The oracle does
    not factor the mean through M-bar, so the linearity of the mean stays a pin and
    is not an assumption.

    """
    w = len(ms)
    p = sum(np.asarray(mw, dtype=np.float64) @ q for mw in ms) / w
    p_hat = orthonormalize(p, orth)
    q_new = sum(np.asarray(mw, dtype=np.float64).T @ p_hat for mw in ms) / w
    q_new = round_to_format(q_new, "f32")
    g_hat = p_hat @ q_new.T
    return PowerStepResult(p=p, p_hat=p_hat, q=q_new, g_hat=g_hat)


def error_update(m_w: np.ndarray, g_hat: np.ndarray, err_fmt: str):
    """E_w = round_E(M_w - G_hat). The buffer keeps what the compressed update left out.

    [card] 证据: billion-parameter stability needs an error buffer. [notes] PowerSGD
    list: the gradient accumulates in the error buffer. Returns (stored E_w, the fp64
    value before rounding).
    """
    pre = np.asarray(m_w, dtype=np.float64) - g_hat
    return round_to_format(pre, err_fmt), pre


# ------------------------------------------------------------------- uncompressed
def uncompressed_mean(u_raw_per_worker, scale: float):
    """Gains and biases: unscale, zero nonfinite, mean over workers, kept in fp32.

    [card] 方法适配: embedding, unembedding, gains and biases are excluded from
    PowerSGD and reduced in 32-bit. [notes] PowerSGD list: they are kept in 32-bit and
    not compressed. The mean is a plain fp64 sum over workers divided by W. [notes]
    Data parallel describes dividing by the worker count before a 16-bit sum. In fp64
    (and in the fp32 the GPU uses) that pre-division does not matter.
    Returns (mean, masks, counts per worker).
    """
    vals, masks, counts = [], [], []
    for u in u_raw_per_worker:
        g, mask = unscale_and_mask(u, scale)
        vals.append(g)
        masks.append(mask)
        counts.append(int(mask.sum()))
    return sum(vals) / len(vals), masks, counts


# --------------------------------------------------------------- whole-block step
@dataclass
class BlockState:
    """Persistent per-block state: E[j][w] (values of the error dtype) and Q[j] (fp32)."""

    e: list  # [J][W] fp64 arrays m_j x n_j
    q: list  # [J] fp64 arrays n_j x r


@dataclass
class BlockResult:
    g_hat: list  # [J] m x n fp64 (zeros when skipped)
    e_pre: list  # [J][W] fp64 pre-rounding E (None when skipped)
    m: list  # [J][W] fp64 values of M (error dtype)
    masks: list  # [J][W] bool
    counts: list  # [W] int: nonfinite entries over the block's matrices and vectors
    skip: bool
    unc_out: np.ndarray | None
    p_hat: list = field(default_factory=list)


def block_step(grads, state: BlockState, scale: float, err_fmt: str,
               skip_fraction: float = 1.0, unc=None, orth: str = "householder"):
    """One PowerSGD step for one resblock: every matrix j, every worker w.

    ``grads[j][w]`` holds the raw (scaled) gradient values as fp64, and ``unc[w]`` the raw
    gains and biases, or None. ``state`` is updated in place unless the block is
    skipped. In that case E and Q are left untouched ([notes] PowerSGD list: the error
    buffer is zeroed as rarely as possible), and G-hat and the gain/bias output are 0.
    """
    J, W = len(grads), len(grads[0])
    ms, masks = [], []
    counts = [0] * W
    numel = 0
    for j in range(J):
        mj, kj = [], []
        for w in range(W):
            g, mask = unscale_and_mask(grads[j][w], scale)
            counts[w] += int(mask.sum())
            mj.append(accumulate_error(g, state.e[j][w], err_fmt))
            kj.append(mask)
        ms.append(mj)
        masks.append(kj)
        numel += grads[j][0].size
    unc_mean = None
    if unc is not None:
        unc_mean, _, uc = uncompressed_mean(unc, scale)
        for w in range(W):
            counts[w] += uc[w]
        numel += np.asarray(unc[0]).size
    skip = skip_block(counts, skip_threshold(skip_fraction, W, numel))
    if skip:
        return BlockResult(
            g_hat=[np.zeros_like(ms[j][0]) for j in range(J)],
            e_pre=[None] * J, m=ms, masks=masks, counts=counts, skip=True,
            unc_out=None if unc is None else np.zeros_like(unc_mean))
    g_hats, e_pres, p_hats = [], [], []
    for j in range(J):
        res = power_step(ms[j], state.q[j], orth)
        state.q[j] = res.q
        pre_j = []
        for w in range(W):
            e_new, pre = error_update(ms[j][w], res.g_hat, err_fmt)
            state.e[j][w] = e_new
            pre_j.append(pre)
        g_hats.append(res.g_hat)
        e_pres.append(pre_j)
        p_hats.append(res.p_hat)
    return BlockResult(g_hat=g_hats, e_pre=e_pres, m=ms, masks=masks, counts=counts,
                       skip=False, unc_out=unc_mean, p_hat=p_hats)


# ------------------------------------------------------------- accounting (closed form)
def compressed_fraction(shapes, rank: int) -> float:
    """Sum over matrices of (m + n) r divided by the sum of m n.

    This is the size of the factors P (m x r) and Q (n x r) sent in place of the m x n
    gradients. [card] 方法适配 and 证据 give a total rank of 896, which is 112 per GPU's
    parameter shard, and about 86% compression. [notes] PowerSGD list gives 85%.
    """
    num = sum((m + n) * rank for m, n in shapes)
    den = sum(m * n for m, n in shapes)
    return num / den
