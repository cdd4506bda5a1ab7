"""Run a workload through the C ABI on the GPU and through the fp64 oracle on the same
seeded inputs, and compare. This is test infrastructure; it is imported only by tests.

Blocks listed in ``oracle_blocks`` get their inputs from ``synth`` on the host, so the
oracle can rebuild them, and are compared. The other blocks of a large workload (the
64-block stack) are filled on the device with torch's seeded normal generator at the
same scale. Blocks are independent, so those values never reach a compared output.
"""
from __future__ import annotations

import concurrent.futures as cf

import numpy as np
import torch

import oracle
import synth

TOL = 1e-4  # relative Frobenius error bound on G-hat and E (fp32 GPU path vs fp64 oracle)
# When the oracle's E is below 2^-20 ||M|| (a planted matrix the step reconstructs), a
# relative bound on E is meaningless: fp32 arithmetic alone leaves O(2^-24 ||M||) there.
# E is then bounded absolutely, ||E_gpu - E_oracle|| <= 2^-18 ||M||.
E_FLOOR, E_ABS = 2.0 ** -20, 2.0 ** -18


def rel_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    nr = float(np.linalg.norm(ref))
    d = float(np.linalg.norm(gpu.astype(np.float64) - ref))
    return d / nr if nr > 0 else d


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


class GpuRun:
    def __init__(self, wl: synth.Workload, oracle_blocks=None, flags: int = 0, device="cuda"):
        from rank_gradient_compression_gb300.psgd import PowerSGD
        self.wl = wl
        self.dev = torch.device(device)
        self.oracle_blocks = list(range(wl.blocks)) if oracle_blocks is None else list(oracle_blocks)
        self.ps = PowerSGD(wl.shapes, wl.blocks, wl.workers, wl.rank, wl.grad_dtype,
                           unc_len=wl.unc_len, skip_fraction=wl.skip_fraction, flags=flags,
                           device=self.dev)
        dt = synth.TORCH_DTYPE[wl.grad_dtype]
        et = synth.TORCH_DTYPE[wl.err_dtype]
        B, W = wl.blocks, wl.workers
        self.grads = [[[torch.empty(s, dtype=dt, device=self.dev) for _ in range(W)] for s in wl.shapes]
                      for _ in range(B)]
        self.errs = [[[torch.zeros(s, dtype=et, device=self.dev) for _ in range(W)] for s in wl.shapes]
                     for _ in range(B)]
        self.q = [[synth.q0(wl, b, j).to(self.dev) for j in range(len(wl.shapes))] for b in range(B)]
        self.ghat = [[torch.empty(s, dtype=torch.float32, device=self.dev) for s in wl.shapes]
                     for _ in range(B)]
        self.unc_in = self.unc_out = None
        if wl.unc_len:
            self.unc_in = [[torch.empty(wl.unc_len, dtype=torch.float32, device=self.dev)
                            for _ in range(W)] for _ in range(B)]
            self.unc_out = [torch.empty(wl.unc_len, dtype=torch.float32, device=self.dev)
                            for _ in range(B)]
        self.scales = [wl.scale(b) for b in range(B)]

    def load_inputs(self, step: int):
        wl = self.wl
        gen = torch.Generator(device=self.dev)
        for b in range(wl.blocks):
            sampled = b in self.oracle_blocks
            if not sampled:
                gen.manual_seed(1_000_003 * step + b)
            for j in range(len(wl.shapes)):
                for w in range(wl.workers):
                    dst = self.grads[b][j][w]
                    if sampled:
                        dst.copy_(synth.grad(wl, step, b, j, w))
                    else:
                        x = torch.randn(dst.shape, generator=gen, device=self.dev, dtype=torch.float32)
                        log2_sig = -12 - 4 * b + (4 * b) % 24 if wl.kind == "stack" else -2
                        dst.copy_((x * 2.0 ** log2_sig).to(dst.dtype))
            if self.unc_in is not None:
                for w in range(wl.workers):
                    self.unc_in[b][w].copy_(synth.unc(wl, step, b, w))

    def step(self):
        self.ps.step(self.grads, self.errs, self.q, self.scales, self.ghat, self.unc_in, self.unc_out)

    def load_state(self, o: "OracleRun"):
        """Overwrite the caller-owned state (E, Q) with the oracle's, so the next step
        starts from identical inputs on both sides. The conversion is exact: the
        oracle holds E-dtype and fp32 values."""
        for b in o.blocks:
            for j in range(len(self.wl.shapes)):
                self.q[b][j].copy_(torch.from_numpy(o.state[b].q[j]).to(torch.float32))
                for w in range(self.wl.workers):
                    self.errs[b][j][w].copy_(torch.from_numpy(o.state[b].e[j][w]).to(self.errs[b][j][w].dtype))


class OracleRun:
    def __init__(self, wl: synth.Workload, blocks, orth="householder"):
        self.wl = wl
        self.blocks = list(blocks)
        self.orth = orth
        self.state = {}
        for b in self.blocks:
            self.state[b] = oracle.BlockState(
                e=[[np.zeros(s) for _ in range(wl.workers)] for s in wl.shapes],
                q=[synth.q0(wl, b, j).double().numpy() for j in range(len(wl.shapes))])

    def step(self, step: int, pool=None, scales=None):
        """One oracle step of every sampled block, unscaled by wl.scale(b), or by
        scales[b] when given (a scale that changes from step to step)."""
        wl = self.wl

        def one(b):
            grads = [[synth.grad(wl, step, b, j, w).double().numpy() for w in range(wl.workers)]
                     for j in range(len(wl.shapes))]
            unc = None
            if wl.unc_len:
                unc = [synth.unc(wl, step, b, w).double().numpy() for w in range(wl.workers)]
            s_b = wl.scale(b) if scales is None else float(scales[b])
            return b, oracle.block_step(grads, self.state[b], s_b, wl.err_dtype,
                                        skip_fraction=wl.skip_fraction, unc=unc, orth=self.orth)

        if pool is None:
            return dict(one(b) for b in self.blocks)
        return dict(pool.map(one, self.blocks))


def _tol(tol, kind, b, j):
    return tol(kind, b, j) if callable(tol) else tol


def compare_step(g: GpuRun, o_res: dict, o: OracleRun, tol=TOL, check_m=True):
    """Compare one step. Returns the worst (G-hat, E before storage, stored E) errors.

    - Masks/counts and skips: bit-exact.
    - M = round_E(g + E): bit-exact when both sides start the step from the same E.
    - G-hat: relative Frobenius error <= tol.
    - E: the value the step computes is M - G-hat, before it is stored in E's type. That
      value is held to tol (absolutely, against ||M||, when the oracle's E is tiny). The
      stored E must be the RNE of the GPU's own M - G-hat, bit for bit: a property of the
      GPU's outputs, checked with the rounding routine. The stored E's distance to the
      oracle's stored E is returned, not asserted. Where G-hat is many times E (a
      decaying spectrum at large r), a G-hat difference far inside tol moves a few
      entries across a 16-bit rounding boundary, and each such entry costs a whole ulp."""
    wl = g.wl
    counts = g.ps.counts.cpu().numpy().reshape(wl.blocks, wl.workers)
    skip = g.ps.skip.cpu().numpy()
    tdt = synth.TORCH_DTYPE[wl.err_dtype]
    worst_g = worst_pre = worst_st = 0.0
    for b, res in o_res.items():
        assert list(counts[b]) == res.counts, f"block {b}: counts {counts[b]} vs {res.counts}"
        assert bool(skip[b]) == res.skip, f"block {b}: skip {skip[b]} vs {res.skip}"
        for j in range(len(wl.shapes)):
            gh = f64(g.ghat[b][j])
            if res.skip:
                assert np.all(gh == 0), f"block {b} matrix {j}: skipped block must give G-hat = 0"
            else:
                eg = rel_err(gh, res.g_hat[j])
                worst_g = max(worst_g, eg)
                assert eg <= _tol(tol, "g", b, j), f"block {b} matrix {j}: G-hat rel err {eg:.3e}"
            for w in range(wl.workers):
                e_gpu = f64(g.errs[b][j][w])
                e_ref = o.state[b].e[j][w]
                m_gpu = f64(g.ps.debug_m(b, j, w, tdt))
                if check_m:
                    assert np.array_equal(m_gpu, res.m[j][w]), f"block {b} matrix {j} worker {w}: M differs"
                if res.skip:
                    assert np.array_equal(e_gpu, e_ref), "skipped block must keep E"
                    continue
                pre_gpu = m_gpu - gh
                assert np.array_equal(e_gpu, oracle.round_to_format(pre_gpu, wl.err_dtype)), \
                    f"block {b} matrix {j} worker {w}: stored E is not RNE(M - G-hat)"
                m_norm = float(np.linalg.norm(res.m[j][w]))
                if float(np.linalg.norm(res.e_pre[j][w])) < E_FLOOR * m_norm:
                    ea = float(np.linalg.norm(pre_gpu - res.e_pre[j][w]))
                    assert ea <= E_ABS * m_norm, f"block {b} matrix {j} worker {w}: |dE| {ea:.3e} vs |M| {m_norm:.3e}"
                else:
                    ep = rel_err(pre_gpu, res.e_pre[j][w])
                    worst_pre = max(worst_pre, ep)
                    assert ep <= _tol(tol, "e", b, j), \
                        f"block {b} matrix {j} worker {w}: E (before storage) rel err {ep:.3e}"
                    worst_st = max(worst_st, rel_err(e_gpu, e_ref))
        if wl.unc_len:
            uo = f64(g.unc_out[b])
            if res.skip:
                assert np.all(uo == 0)
            else:
                # The output is fp32, so the oracle's mean is compared after its own rounding
                # to fp32. Terms below fp32's range (deep blocks of the stack) underflow on
                # both sides; the floor allows one subnormal ulp per worker and entry.
                ref = oracle.round_to_format(res.unc_out, "f32")
                utol = TOL if callable(tol) else tol
                du = float(np.linalg.norm(uo - ref))
                floor = wl.workers * 2.0 ** -149 * np.sqrt(ref.size)
                assert du <= utol * float(np.linalg.norm(ref)) + floor, \
                    f"block {b}: gains/biases error {du:.3e} (|ref| {np.linalg.norm(ref):.3e})"
    return worst_g, worst_pre, worst_st


def ulp_diff(a: torch.Tensor, b: np.ndarray) -> int:
    """Largest distance in units in the last place between two arrays of a 16-bit or
    fp32 type (finite values; same-sign ordering of the bit patterns)."""
    dt = a.dtype
    bt = torch.from_numpy(b).to(dt)
    it = {torch.float16: torch.int16, torch.bfloat16: torch.int16, torch.float32: torch.int32}[dt]
    ia = a.detach().cpu().view(it).to(torch.int64)
    ib = bt.view(it).to(torch.int64)
    sign = 1 << (15 if it == torch.int16 else 31)
    # map sign-magnitude bit patterns onto a monotone integer line
    ia = torch.where(ia < 0, -(ia + sign), ia)
    ib = torch.where(ib < 0, -(ib + sign), ib)
    return int((ia - ib).abs().max().item())


def run_parity(wl, steps=None, oracle_blocks=None, flags=0, tol=TOL, check_m=True, threads=8,
               synced=True):
    """Run both sides over the steps and compare each step.

    synced=True (default) copies the oracle's E and Q into the GPU's caller-owned buffers
    before every step. Each step then starts from identical inputs, and M is compared bit
    for bit every step. The maximum one-ulp distance of the stored E is reported by
    ulp_diff, not asserted: where E is near zero, a G-hat difference far below E's
    tolerance can span several of E's ulps. With synced=False each side carries its own state. The warm-started power
    iteration then amplifies the one-ulp differences of the stored E into a growing
    rotation of the subspace wherever singular-value gaps are small. That is the
    method's sensitivity, not kernel error, and only the first step is compared at the
    1e-4 bar in that mode."""
    steps = wl.steps if steps is None else steps
    g = GpuRun(wl, oracle_blocks, flags)
    o = OracleRun(wl, g.oracle_blocks)
    worst = []
    with cf.ThreadPoolExecutor(threads) as pool:
        for t in range(steps):
            g.load_inputs(t)
            if synced:
                g.load_state(o)
            g.step()
            torch.cuda.synchronize()
            res = o.step(t, pool)
            worst.append(compare_step(g, res, o, tol, check_m and (synced or t == 0)))
    return g, o, worst
