"""psgd_orthonormalize_static: the orthonormalisation of one P with the library's fixed
scratch array, for callers that cannot allocate.

It is compared with the orthonormalisation inside psgd_step (the P^ that step leaves
behind, read through psgd_debug_phat) on the P of that same step, and with the oracle's
Householder basis, on two calls in a row. This file is collected last, and it also
passes on its own in a fresh process (the first call on a device does the set-up).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from harness import GpuRun, TOL, f64, rel_err

pytestmark = pytest.mark.gpu


def _psgd():
    from rank_gradient_compression_gb300 import psgd
    return psgd


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _static(psgd, p: torch.Tensor) -> torch.Tensor:
    m, r = p.shape
    out = torch.full((m, r), float("nan"), dtype=torch.float32, device=p.device)
    psgd.psgd_orthonormalize_static(p.data_ptr(), out.data_ptr(), m, r, _stream())
    return out


def _projector_err(ph: np.ndarray, p: np.ndarray) -> float:
    """Relative error of ph ph^T against the oracle's projector onto span(p), applied to
    a fixed random probe (an m x m projector is not formed)."""
    qo = oracle.orthonormalize(p)
    z = np.random.default_rng(7).standard_normal((p.shape[0], 8))
    return rel_err(ph @ (ph.T @ z), qo @ (qo.T @ z))


def _check_basis(ph: np.ndarray):
    gram = ph.T @ ph
    assert np.abs(gram - np.eye(gram.shape[0])).max() <= 1e-5


def test_static_orth_matches_the_step_orth_two_calls_in_a_row():
    """Two steps of a ragged fp16 workload (m not a multiple of 64, r = 40 not a multiple
    of 16). After each step, P = (1/W) sum_w M_w Q is rebuilt from the step's own M
    scratch and its input Q (fp64, rounded to fp32). The static entry point is called
    twice in a row on it: both results are identical, they match the step's P^ within
    the parity tolerance, and they span the oracle's span(P)."""
    psgd = _psgd()
    wl = synth.with_shapes(synth.resblock_shard(steps=2, workers=3, rank=40),
                           ((1000, 304), (2100, 144)))
    g = GpuRun(wl)
    for t in range(wl.steps):
        g.load_inputs(t)
        q_in = [q.clone() for q in g.q[0]]
        g.step()
        g.ps.check()
        for j, (m, n) in enumerate(wl.shapes):
            ms = [g.ps.debug_m(0, j, w, torch.float16).to(torch.float64) for w in range(wl.workers)]
            p64 = sum(mw @ q_in[j].to(torch.float64) for mw in ms) / wl.workers
            p = p64.to(torch.float32).contiguous()
            first = _static(psgd, p)
            second = _static(psgd, p)
            step_phat = g.ps.debug_phat(0, j).clone()
            torch.cuda.synchronize()
            assert torch.equal(first, second), (t, j)
            a = f64(first)
            assert np.isfinite(a).all()
            e_step = rel_err(a, f64(step_phat))
            e_orc = _projector_err(a, f64(p))
            print(f"step {t} matrix {j}: vs psgd_step P^ {e_step:.2e}, vs oracle span {e_orc:.2e}")
            assert e_step <= TOL, (t, j, e_step)
            assert e_orc <= TOL, (t, j, e_orc)
            _check_basis(a)


def test_static_orth_at_the_size_limit_allocates_nothing():
    """m = 16384 rows and r = 128 columns (the limits), then a smaller ragged matrix,
    then the limit again: each result spans span(P) and is orthonormal, and the device's
    free memory is the same before and after the calls."""
    psgd = _psgd()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(11)
    big = torch.randn((psgd.PSGD_STATIC_MAX_ROWS, psgd.PSGD_STATIC_MAX_COLS), generator=gen,
                      device="cuda")
    small = torch.randn((777, 19), generator=gen, device="cuda") * 2.0 ** -70
    outs = [torch.empty_like(big), torch.empty_like(small), torch.empty_like(big)]
    ins = [big, small, big]
    # warm-up call: the first call on the device looks up the scratch address
    psgd.psgd_orthonormalize_static(small.data_ptr(), outs[1].data_ptr(), 777, 19, _stream())
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for x, y in zip(ins, outs):
        psgd.psgd_orthonormalize_static(x.data_ptr(), y.data_ptr(), x.shape[0], x.shape[1],
                                        _stream())
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    assert torch.equal(outs[0], outs[2])
    for x, y in zip(ins[:2], outs[:2]):
        a = f64(y)
        assert _projector_err(a, f64(x)) <= TOL
        _check_basis(a)


def test_static_orth_rejects_sizes_beyond_the_limit():
    psgd = _psgd()
    lim_m, lim_r = psgd.PSGD_STATIC_MAX_ROWS, psgd.PSGD_STATIC_MAX_COLS
    buf = torch.zeros(2 * (lim_m + 1) * (lim_r + 1), dtype=torch.float32, device="cuda")
    half = buf.numel() // 2
    a, b = buf.data_ptr(), buf[half:].data_ptr()
    cases = [((lim_m + 1, 8), "16384 rows"), ((64, lim_r + 1), "128 columns"),
             ((10, 11), "r must be <= m"), ((0, 1), ">= 1")]
    for (m, r), words in cases:
        with pytest.raises(psgd.PSGDError) as ex:
            psgd.psgd_orthonormalize_static(a, b, m, r, _stream())
        assert ex.value.status == psgd.PSGD_EINVAL
        assert words in str(ex.value), str(ex.value)
    with pytest.raises(psgd.PSGDError) as ex:  # overlapping input and output
        psgd.psgd_orthonormalize_static(a, a + 4 * 64, 128, 8, _stream())
    assert ex.value.status == psgd.PSGD_EINVAL
    with pytest.raises(psgd.PSGDError) as ex:
        psgd.psgd_orthonormalize_static(0, b, 16, 4, _stream())
    assert ex.value.status == psgd.PSGD_EINVAL


def test_static_orth_accepts_4_byte_aligned_pointers():
    """The entry point promises only 4-byte alignment. With both pointers 4 bytes off a
    16-byte boundary (r a multiple of 4, so only the pointers rule out 16-byte accesses),
    the result equals the one from aligned buffers bit for bit."""
    psgd = _psgd()
    m, r = 1000, 40
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    p = torch.randn((m, r), generator=gen, device="cuda")
    ref = _static(psgd, p)
    pbuf = torch.zeros(m * r + 4, device="cuda")
    obuf = torch.full((m * r + 4,), float("nan"), device="cuda")
    pv = pbuf[1:1 + m * r]
    pv.copy_(p.reshape(-1))
    ov = obuf[1:1 + m * r]
    psgd.psgd_orthonormalize_static(pv.data_ptr(), ov.data_ptr(), m, r, _stream())
    torch.cuda.synchronize()
    assert pv.data_ptr() % 16 == 4 and ov.data_ptr() % 16 == 4
    assert torch.equal(ov.view(m, r), ref)
