"""Seeded synthetic workloads for the PowerSGD step (shared by the tests, the bench and
the oracle's callers).

This module holds shapes, seeds and random draws only. None of the step's arithmetic
is here. Every draw comes from numpy's PCG64, seeded through SeedSequence with the key
(base seed, workload tag, step, block, matrix, worker, stream). Any block of any step
can therefore be regenerated on its own, on any machine, without holding the
workload's other blocks.

The shapes are those of one 8-way column shard of a resblock of the 12B DALL·E
transformer (d_model = 3968; "Zero-Shot Text-to-Image Generation - 中文验证版",
§计算设置 and §方法适配): qkv 3968x1488, attn-out 3968x496, mlp-in 3968x1984 and
mlp-out 15872x496.

Raw gradients are returned as CPU torch tensors in their storage dtype. A value is
drawn in fp64, rounded to fp32, then converted with torch to fp16/bf16 (RNE). That
conversion defines the raw input; both the oracle and the GPU read the same tensor.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from functools import lru_cache

import numpy as np
import torch

BASE_SEED = 20210224
D_MODEL = 3968
SHARD_SHAPES = ((3968, 1488), (3968, 496), (3968, 1984), (15872, 496))
SHARD_NAMES = ("qkv", "attn_out", "mlp_in", "mlp_out")

TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}

_TAGS = {}


def _tag(name: str) -> int:
    if name not in _TAGS:
        _TAGS[name] = int.from_bytes(name.encode()[:8].ljust(8, b"\0"), "little") & 0x7FFFFFFF
    return _TAGS[name]


@dataclass(frozen=True)
class Workload:
    """One synthetic workload. ``kind`` selects the gradient recipe."""

    name: str
    kind: str  # "gauss" | "planted" | "stack" | "spectrum" | "stress"
    shapes: tuple
    blocks: int
    workers: int
    rank: int
    grad_dtype: str
    err_dtype: str
    steps: int
    unc_len: int = 0
    sigma_raw: float = 2.0 ** -2  # std of the raw (scaled) gradient
    scale_log2: int = 10  # s_b = 2**scale_log2 (block-constant kinds)
    skip_fraction: float = 1.0
    params: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def numel_block(self) -> int:
        return sum(m * n for m, n in self.shapes) + self.unc_len

    def scale(self, block: int) -> float:
        if self.kind == "stack":
            return 2.0 ** ((4 * block) % 24)
        return 2.0 ** self.scale_log2

    def grad_bytes_per_step(self) -> int:
        esz = {"f32": 4, "f16": 2, "bf16": 2}[self.grad_dtype]
        return self.blocks * self.workers * sum(m * n for m, n in self.shapes) * esz


def fp32_small(m=256, n=512, rank=4, workers=2, steps=1):
    """A single fp32 256x512 gradient matrix, N(0, 1e-3) entries (std 1e-3), r = 4,
    W = 2, s_b = 1, and one step."""
    return Workload("fp32_256x512_r4_w2", "gauss", ((m, n),), 1, workers, rank, "f32",
                    "f32", steps, sigma_raw=1e-3, scale_log2=0)


def planted_rank3(m=256, n=512, rank=4, workers=2):
    """An fp32 U V^T matrix of rank 3 (U: m x 3, V: n x 3). U and V are N(0,1) rounded
    to multiples of 2^-6, so every entry of U V^T is exact in fp32 and the matrix has
    rank exactly 3. Both workers hold the same matrix."""
    return Workload("planted_rank3_256x512_r4_w2", "planted", ((m, n),), 1, workers, rank,
                    "f32", "f32", 1, scale_log2=0)


def resblock_shard(steps=10, workers=8, rank=112, shapes=SHARD_SHAPES, blocks=1,
                   dtype="f16"):
    """One resblock shard (the four matrices above), fp16 raw N(0, 2^-2): that is
    sigma = 2^-12 times s_b = 2^10. Fresh gradients every step, W = 8, r = 112."""
    return Workload(f"resblock_shard_{dtype}_w{workers}_r{rank}", "gauss", tuple(shapes),
                    blocks, workers, rank, dtype, dtype, steps)


def stack64(steps=2, workers=4, rank=112, blocks=64, shapes=SHARD_SHAPES):
    """64 resblock shards in bf16 with W = 4 and r = 112. The true gradient of block b
    has std 2^-12 * 2^(-4b), and the scale is s_b = 2^(4b mod 24). The raw value is
    bf16(fp32(true * s_b)), so deep blocks underflow to subnormals and then to zero.
    Gains and biases are 2 x 3968 fp32 per block per worker, drawn the same way."""
    return Workload(f"stack{blocks}_bf16_w{workers}_r{rank}", "stack", tuple(shapes), blocks,
                    workers, rank, "bf16", "bf16", steps, unc_len=2 * D_MODEL)


def spectrum(rank=112, steps=5, m=3968, n=15872, workers=8):
    """One fp16 3968x15872 gradient U diag(c/k) V^T. U and V are orthonormal, from fp64
    QR of Gaussians. c makes the raw RMS 2^-2 at s_b = 2^10. Every worker holds the
    same matrix, and the same gradient is fed at every step."""
    return Workload(f"spectrum_{m}x{n}_fp16_w{workers}_r{rank}", "spectrum", ((m, n),), 1,
                    workers, rank, "f16", "f16", steps)


def stress(steps=3, workers=8, rank=112, blocks=2, shapes=SHARD_SHAPES, bad_block=1,
           bad_step=1, frac=1e-3):
    """Resblock-shard shapes in fp16. |v| is log-uniform in [2^-30, 2^0] with random
    signs, and raw = fp16(v * 2^10). At seeded positions, a fraction 1e-3 of each
    (matrix, worker) is set to +Inf/-Inf/NaN in equal thirds. Block ``bad_block`` is
    entirely nonfinite at step ``bad_step`` on every worker."""
    return Workload(f"stress_fp16_w{workers}_r{rank}", "stress", tuple(shapes), blocks,
                    workers, rank, "f16", "f16", steps,
                    params={"bad_block": bad_block, "bad_step": bad_step, "frac": frac})


def scaler_run(steps=5, workers=2, rank=8, shapes=((256, 192), (96, 64)),
               spots=((1, 1, 5), (3, 0, 1))):
    """Two blocks in fp16 for the dynamic-scale test: stress-style magnitudes with no
    random nonfinite entries, except at the (step, block, count) spots, where matrix 0
    of worker 0 gets `count` nonfinite entries (Inf, -Inf, NaN in thirds) at seeded
    positions."""
    return Workload(f"scaler_fp16_w{workers}_r{rank}", "stress", tuple(shapes), 2, workers,
                    rank, "f16", "f16", steps,
                    params={"frac": 0.0, "spots": {(st, b): c for st, b, c in spots}})


def with_shapes(wl: Workload, shapes, **kw) -> Workload:
    return replace(wl, shapes=tuple(shapes), **kw)


# ------------------------------------------------------------------------ draws
def _rng(wl: Workload, *key) -> np.random.Generator:
    return np.random.default_rng([BASE_SEED, _tag(wl.kind), *[int(k) for k in key]])


def _to_storage(x64: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x64, dtype=np.float64).astype(np.float32))
    return t.to(TORCH_DTYPE[dtype]).contiguous()


@lru_cache(maxsize=2)
def _spectrum_base(m: int, n: int) -> np.ndarray:
    rng = np.random.default_rng([BASE_SEED, _tag("spectrum"), m, n])
    k = min(m, n)
    u, _ = np.linalg.qr(rng.standard_normal((m, k)))
    v, _ = np.linalg.qr(rng.standard_normal((n, k)))
    sig = 1.0 / np.arange(1, k + 1, dtype=np.float64)
    c = 2.0 ** -2 * math.sqrt(m * n) / math.sqrt(float(np.sum(sig ** 2)))
    g = (u * (c * sig)) @ v.T
    return g


def spectrum_singular_values(wl: Workload) -> np.ndarray:
    """The designed singular values of the raw spectrum gradient (before fp16 rounding)."""
    m, n = wl.shapes[0]
    k = min(m, n)
    sig = 1.0 / np.arange(1, k + 1, dtype=np.float64)
    c = 2.0 ** -2 * math.sqrt(m * n) / math.sqrt(float(np.sum(sig ** 2)))
    return c * sig


def _planted(wl: Workload, m: int, n: int) -> np.ndarray:
    rng = _rng(wl, 0, 0, 0, 0, 7)
    u = np.round(rng.standard_normal((m, 3)) * 64.0) / 64.0
    v = np.round(rng.standard_normal((n, 3)) * 64.0) / 64.0
    return u @ v.T


def grad(wl: Workload, step: int, block: int, j: int, w: int) -> torch.Tensor:
    """Raw (scaled) gradient of worker w, matrix j, block b at a step: m x n, row-major."""
    m, n = wl.shapes[j]
    if wl.kind == "gauss":
        x = _rng(wl, step, block, j, w, 0).standard_normal((m, n)) * wl.sigma_raw
    elif wl.kind == "planted":
        x = _planted(wl, m, n)
    elif wl.kind == "stack":
        log2_sig = -12 - 4 * block + (4 * block) % 24
        x = _rng(wl, step, block, j, w, 0).standard_normal((m, n)) * 2.0 ** log2_sig
    elif wl.kind == "spectrum":
        x = _spectrum_base(m, n)
    elif wl.kind == "stress":
        x = _stress_values(wl, step, block, j, w, m, n)
    else:
        raise ValueError(wl.kind)
    return _to_storage(x, wl.grad_dtype)


def _stress_values(wl, step, block, j, w, m, n):
    rng = _rng(wl, step, block, j, w, 0)
    mag = 2.0 ** rng.uniform(-30.0, 0.0, size=(m, n))
    sgn = np.where(rng.random((m, n)) < 0.5, -1.0, 1.0)
    x = sgn * mag * 2.0 ** wl.scale_log2
    p = wl.params
    if block == p.get("bad_block", -1) and step == p.get("bad_step", -1):
        kinds = rng.integers(0, 3, size=(m, n))
        return np.choose(kinds, [np.inf, -np.inf, np.nan]).astype(np.float64)
    cnt = int(round(p.get("frac", 1e-3) * m * n))
    if j == 0 and w == 0:
        cnt += p.get("spots", {}).get((step, block), 0)
    pos = rng.choice(m * n, size=cnt, replace=False)
    flat = x.reshape(-1)
    third = cnt // 3
    flat[pos[:third]] = np.inf
    flat[pos[third:2 * third]] = -np.inf
    flat[pos[2 * third:]] = np.nan
    return x


def unc(wl: Workload, step: int, block: int, w: int):
    """Raw gains and biases of worker w (fp32, unc_len entries) or None."""
    if wl.unc_len == 0:
        return None
    log2_sig = -12 - 4 * block + (4 * block) % 24 if wl.kind == "stack" else -2
    x = _rng(wl, step, block, 99, w, 1).standard_normal(wl.unc_len) * 2.0 ** log2_sig
    return _to_storage(x, "f32")


def q0(wl: Workload, block: int, j: int) -> torch.Tensor:
    """Initial Q (n x r, fp32), N(0, 1). It is the same on both sides and is passed in."""
    n = wl.shapes[j][1]
    x = _rng(wl, 0, block, j, 0, 2).standard_normal((n, wl.rank))
    return torch.from_numpy(x.astype(np.float32))


def zeros_err(wl: Workload, j: int) -> torch.Tensor:
    m, n = wl.shapes[j]
    return torch.zeros((m, n), dtype=TORCH_DTYPE[wl.err_dtype])


# ------------------------------------------------------------- uncompressed tensors
# The image vocabulary is 8192 and the transformer sees 256 text + 1024 image positions
# with d_model = 3968 ("Zero-Shot Text-to-Image Generation - 中文验证版", §计算设置). The
# pages do not give the text vocabulary, so the vocabulary-scale tensor here is the image
# embedding (8192 x 3968); the unembedding has the same shape.
IMAGE_VOCAB = 8192


def embedding_grad(step: int, w: int, rows: int = IMAGE_VOCAB, cols: int = D_MODEL,
                   log2_sig: int = -2, frac: float = 1e-3, scale_log2: int = 10) -> torch.Tensor:
    """Raw (scaled) fp32 gradient of a vocabulary x d_model embedding on worker w, flattened:
    N(0, 2^log2_sig) values (the true gradient times 2^scale_log2), and a fraction `frac`
    of the entries at seeded positions set to +Inf, -Inf and NaN in thirds."""
    rng = np.random.default_rng([BASE_SEED, _tag("embed"), step, rows, cols, w, scale_log2])
    n = rows * cols
    x = rng.standard_normal(n, dtype=np.float32) * np.float32(2.0 ** log2_sig)
    cnt = int(round(frac * n))
    pos = rng.choice(n, size=cnt, replace=False)
    third = cnt // 3
    x[pos[:third]] = np.inf
    x[pos[third:2 * third]] = -np.inf
    x[pos[2 * third:]] = np.nan
    return torch.from_numpy(x)
