"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bars: masks, nonfinite counts, skip decisions and M are bit-exact. G-hat and E are
within 1e-4 relative Frobenius error per matrix, the fp32 GPU path against the fp64
oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import numerics as nx
from harness import GpuRun, OracleRun, TOL, compare_step, f64, rel_err, run_parity

pytestmark = pytest.mark.gpu


def _psgd():
    from rank_gradient_compression_gb300 import psgd
    return psgd


# ------------------------------------------------------------------ ingest brute force
@pytest.mark.parametrize("dtype,scale", [("f16", 2.0 ** 10), ("bf16", 2.0 ** 20), ("f16", 1.0)])
def test_ingest_every_bit_pattern(dtype, scale):
    """Every 16-bit pattern as a gradient entry, under random finite error-buffer values.
    M, the mask bitmap and the counts must equal the oracle's bit for bit."""
    psgd = _psgd()
    tdt = synth.TORCH_DTYPE[dtype]
    rng = np.random.default_rng(11)
    W, m, n = 2, 256, 256
    ps = psgd.PowerSGD([(m, n)], 1, W, 1, dtype, flags=psgd.PSGD_FLAG_MASK | psgd.PSGD_FLAG_STOP_AFTER_INGEST)
    grads, errs, gin, ein = [], [], [], []
    for w in range(W):
        bits = rng.permutation(1 << 16).astype(np.uint16)
        gt = torch.from_numpy(bits.view(np.int16).reshape(m, n)).view(tdt)
        eb = rng.integers(0, 0x7C00 if dtype == "f16" else 0x7F80, size=m * n).astype(np.uint16)
        eb |= (rng.random(m * n) < 0.5).astype(np.uint16) << 15
        et = torch.from_numpy(eb.view(np.int16).reshape(m, n)).view(tdt)
        grads.append(gt.cuda()); errs.append(et.cuda())
        gin.append(gt.to(torch.float64).numpy()); ein.append(et.to(torch.float64).numpy())
    q = [[torch.zeros((n, 1), device="cuda")]]
    gh = [[torch.zeros((m, n), device="cuda")]]
    ps.step([[grads]], [[errs]], q, [scale], gh)
    torch.cuda.synchronize()
    counts = ps.counts.cpu().numpy()
    masks = ps.mask.cpu().numpy().view(np.uint8)
    for w in range(W):
        g, mask = oracle.unscale_and_mask(gin[w], scale)
        want_m = oracle.accumulate_error(g, ein[w], dtype)
        got_m = f64(ps.debug_m(0, 0, w, tdt))
        same = (got_m == want_m) | (np.isnan(got_m) & np.isnan(want_m))
        assert same.all(), f"worker {w}: {int((~same).sum())} M entries differ"
        assert counts[w] == int(mask.sum())
        off = psgd.psgd_mask_offset(ps.cfg, 0, 0, w) * 4
        want_bits = np.packbits(mask.reshape(-1), bitorder="little")
        assert np.array_equal(masks[off:off + want_bits.size], want_bits)
    assert counts.sum() == 2 * (2048 if dtype == "f16" else 256)  # all-ones exponent patterns


@pytest.mark.parametrize("dtype,scale", [("f16", 2.0 ** 10), ("f16", 1.0), ("f16", 2.0 ** 20),
                                         ("bf16", 2.0 ** 20)])
def test_fused_ingest_every_bit_pattern(dtype, scale):
    """The production path (the fused ingest + P GEMM kernel, a full step): every 16-bit
    pattern once per worker as a gradient entry, under random finite error-buffer values
    below 2^10. M, the nonfinite mask bitmap and the counts must equal the oracle's bit
    for bit."""
    psgd = _psgd()
    tdt = synth.TORCH_DTYPE[dtype]
    rng = np.random.default_rng(13)
    W, m, n, r = 2, 256, 256, 16
    ps = psgd.PowerSGD([(m, n)], 1, W, r, dtype, flags=psgd.PSGD_FLAG_MASK)
    assert ps.engine == "tcgen05"
    grads, errs, gin, ein = [], [], [], []
    top = 0x6400 if dtype == "f16" else 0x4480  # |E| < 2^10
    for w in range(W):
        bits = rng.permutation(1 << 16).astype(np.uint16)
        gt = torch.from_numpy(bits.view(np.int16).reshape(m, n)).view(tdt)
        eb = rng.integers(0, top, size=m * n).astype(np.uint16)
        eb |= (rng.random(m * n) < 0.5).astype(np.uint16) << 15
        et = torch.from_numpy(eb.view(np.int16).reshape(m, n)).view(tdt)
        grads.append(gt.cuda()); errs.append(et.cuda())
        gin.append(gt.to(torch.float64).numpy()); ein.append(et.to(torch.float64).numpy())
    q = [[torch.from_numpy(rng.standard_normal((n, r)).astype(np.float32)).cuda()]]
    gh = [[torch.zeros((m, n), device="cuda")]]
    ps.step([[grads]], [[errs]], q, [scale], gh)
    torch.cuda.synchronize()
    counts = ps.counts.cpu().numpy()
    for w in range(W):
        g, mask = oracle.unscale_and_mask(gin[w], scale)
        want_m = oracle.accumulate_error(g, ein[w], dtype)
        got_m = f64(ps.debug_m(0, 0, w, tdt))
        same = (got_m == want_m) | (np.isnan(got_m) & np.isnan(want_m))
        assert same.all(), f"worker {w}: {int((~same).sum())} M entries differ"
        assert counts[w] == int(mask.sum())
        off = psgd.psgd_mask_offset(ps.cfg, 0, 0, w)
        words = ps.mask[off:off + m * n // 32].cpu().numpy().astype(np.uint32)
        got_mask = np.unpackbits(words.view(np.uint8), bitorder="little").astype(bool)
        assert np.array_equal(got_mask, mask.reshape(-1)), f"worker {w}: mask bits differ"


def test_ingest_fp32_specials():
    psgd = _psgd()
    rng = np.random.default_rng(12)
    m, n = 64, 128
    bits = rng.integers(0, 2 ** 32, size=m * n, dtype=np.uint64).astype(np.uint32)
    bits[:64] = [0x7F800000, 0xFF800000, 0x7FC00000, 0x00000001, 0x80000001, 0x7F7FFFFF] * 10 + [0, 0x80000000, 1, 2]
    g = torch.from_numpy(bits.view(np.float32).reshape(m, n).copy())
    e = torch.from_numpy((rng.standard_normal((m, n)) * 1e-3).astype(np.float32))
    ps = psgd.PowerSGD([(m, n)], 1, 1, 1, "f32", flags=psgd.PSGD_FLAG_MASK | psgd.PSGD_FLAG_STOP_AFTER_INGEST)
    ps.step([[[g.cuda()]]], [[[e.cuda()]]], [[torch.zeros((n, 1), device="cuda")]], [4.0],
            [[torch.zeros((m, n), device="cuda")]])
    torch.cuda.synchronize()
    gg, mask = oracle.unscale_and_mask(g.double().numpy(), 4.0)
    want = oracle.accumulate_error(gg, e.double().numpy(), "f32")
    got = f64(ps.debug_m(0, 0, 0, torch.float32))
    assert np.array_equal(got, want)
    assert int(ps.counts.cpu()[0]) == int(mask.sum())


# ------------------------------------------------------------------ whole-step parity
def test_fp32_small_one_step():
    """Small fp32 case: a 256x512 matrix, N(0, 1e-3), r = 4, W = 2, one step."""
    _, _, worst = run_parity(synth.fp32_small())
    assert worst[0][0] <= TOL


def test_planted_rank3_reconstructs():
    """The planted U V^T of rank 3 at r = 4: G-hat = M within 1e-5 on the GPU, and the
    mean error buffer is ~0."""
    wl = synth.planted_rank3()
    g, o, _ = run_parity(wl)
    m = synth.grad(wl, 0, 0, 0, 0).double().numpy()
    assert rel_err(f64(g.ghat[0][0]), m) <= 1e-5
    e = sum(f64(g.errs[0][0][w]) for w in range(wl.workers)) / wl.workers
    assert np.linalg.norm(e) <= 1e-5 * np.linalg.norm(m)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("shapes,W,r", [
    (((200, 136), (64, 40)), 3, 4),
    (((333, 264),), 2, 16),
    (((130, 72), (257, 520)), 1, 1),
    (((256, 512), (384, 128)), 8, 32),
    (((300, 264), (130, 136)), 2, 124),
    (((700, 600),), 2, 200),
])
def test_small_ragged_multi_step(dtype, shapes, W, r):
    """Ragged shapes (not multiples of any tile), three steps with fresh gradients. r = 124
    has more than 128 8 x 8 blocks in the Gram upper triangle; r = 200 runs the FFMA engine
    and orthonormalises in two column blocks (128 + 72)."""
    wl = synth.with_shapes(synth.resblock_shard(steps=3, workers=W, rank=r, dtype=dtype), shapes)
    run_parity(wl)


def test_simt_engine_matches_default_engine():
    """The FFMA debug engine and the default engine agree to the same oracle."""
    psgd = _psgd()
    wl = synth.with_shapes(synth.resblock_shard(steps=2, workers=2, rank=8), ((256, 192),))
    run_parity(wl, flags=psgd.PSGD_FLAG_SIMT)


def test_resblock_shard_full_size_ten_steps():
    """One d_model = 3968 resblock shard: fp16, W = 8, r = 112, ten steps. This is the
    workload that bench.py times, at full size."""
    _, _, worst = run_parity(synth.resblock_shard(steps=10))
    print("worst (G-hat, E) per step:", worst)


def test_free_running_first_step_and_drift():
    """Without resynchronisation, the first step is held to the 1e-4 bar. Later steps are
    only reported: each side's own rounding feeds its next step."""
    _, _, worst = run_parity(synth.with_shapes(synth.resblock_shard(steps=3, workers=4, rank=16),
                                               ((512, 256), (256, 512))), synced=False, tol=1.0)
    assert worst[0][0] <= TOL and worst[0][1] <= TOL
    print("free-running (G-hat, E) per step:", worst)


def test_stress_nonfinite_and_skip():
    """Log-uniform magnitudes across the fp16 subnormal range, 0.1% of entries +-Inf/NaN,
    block 1 fully nonfinite at step 1: bit-exact masks/counts/skips, and block 1 keeps
    E and Q bit-for-bit through the faulted step."""
    wl = synth.stress()
    g = GpuRun(wl)
    o = OracleRun(wl, range(wl.blocks))
    for t in range(wl.steps):
        g.load_inputs(t)
        g.load_state(o)
        e_before = [[g.errs[1][j][w].clone() for w in range(wl.workers)] for j in range(4)]
        q_before = [g.q[1][j].clone() for j in range(4)]
        g.step()
        torch.cuda.synchronize()
        res = o.step(t)
        compare_step(g, res, o, check_m=True)
        skip = g.ps.skip.cpu().numpy()
        assert bool(skip[1]) == (t == 1) and not skip[0]
        if t == 1:
            for j in range(4):
                assert torch.equal(g.q[1][j], q_before[j])
                for w in range(wl.workers):
                    assert torch.equal(g.errs[1][j][w], e_before[j][w])


def test_stack64_sampled_blocks():
    """64 resblock shards (bf16, W = 4, r = 112, per-block scales 2^(4b mod 24), fp32
    gains/biases) in one call. The oracle checks sampled blocks, among them blocks whose
    gradients are subnormal or all zero."""
    wl = synth.stack64()
    run_parity(wl, oracle_blocks=[0, 5, 6, 17, 30, 35, 36, 63])


@pytest.mark.parametrize("rank", [16, 32, 64, 112, 256, 640, 896])
def test_spectrum_rank_sweep(rank):
    """3968x15872 fp16 gradient with singular values c/k, W = 8 identical copies, 5 steps.
    Ranks above 128 run on the FFMA engine with the orthonormalisation in 128-column
    blocks (block Gram-Schmidt with re-orthogonalisation, CholeskyQR within a block).

    After the first warm start, P has condition number about 1.5e6 at r = 896 and its
    columns, scaled to unit length, about 4e5. G-hat and E (before storage) are held to
    the plain 1e-4 at every rank and step. Holding P in fp32 already costs about 4e-5 of
    E at r = 896 there; the products that change the span of P (X R^-1 and the block
    projections) are compensated so that the orthonormalisation adds little to it."""
    wl = synth.spectrum(rank=rank, steps=5)
    g = GpuRun(wl)
    o = OracleRun(wl, [0])
    for t in range(wl.steps):
        g.load_inputs(t)
        g.load_state(o)
        g.step()
        torch.cuda.synchronize()
        res = o.step(t)
        errs = compare_step(g, res, o)
        print(f"rank {rank} step {t}: GPU (G-hat, E, stored E) {errs}")


# ------------------------------------------------------------------ properties
def test_orthonormal_basis_and_ef_identity():
    wl = synth.with_shapes(synth.resblock_shard(steps=1, workers=3, rank=24), ((700, 312), (1024, 96)))
    g, o, _ = run_parity(wl)
    for j, (m, n) in enumerate(wl.shapes):
        ph = f64(g.ps.debug_phat(0, j))
        live = np.linalg.norm(ph, axis=0) > 0.5
        gram = ph[:, live].T @ ph[:, live]
        assert np.abs(gram - np.eye(int(live.sum()))).max() <= 1e-5
        # M_w = G-hat + E_w up to the rounding of E (half an ulp of E's type, RNE)
        gh = f64(g.ghat[0][j])
        for w in range(wl.workers):
            mm = f64(g.ps.debug_m(0, j, w, torch.float16))
            ee = f64(g.errs[0][j][w])
            assert np.array_equal(ee, nx.round_to_format(ee, "f16"))
            assert np.abs(mm - gh - ee).max() <= 2.0 ** -11 * np.abs(mm - gh).max() + 1e-12


def test_orth_pass_counts():
    """The adaptive CholeskyQR needs at most two passes on well-conditioned P (random
    gradients). The planted rank-deficient case needs shifted passes. Both end with an
    orthonormal basis of span(P)."""
    wl = synth.with_shapes(synth.resblock_shard(steps=2, workers=2, rank=16), ((512, 256),))
    g, o, _ = run_parity(wl)
    n, rec = g.ps.debug_orth(0, 0)
    assert 1 <= n <= 2, rec
    gp, _, _ = run_parity(synth.planted_rank3())
    n2, rec2 = gp.ps.debug_orth(0, 0)
    assert n2 >= 2 and rec2[0][2] == 1, rec2  # the first pass was shifted


def test_deterministic_and_resumable():
    """Two runs give bit-identical outputs. Four straight steps equal two steps, a
    save/restore of the caller-owned state (E, Q) into fresh buffers and a fresh
    handle, and two more steps."""
    wl = synth.with_shapes(synth.resblock_shard(steps=4, workers=2, rank=8), ((256, 128),))
    a = GpuRun(wl)
    for t in range(4):
        a.load_inputs(t); a.step()
    b = GpuRun(wl)
    for t in range(2):
        b.load_inputs(t); b.step()
    torch.cuda.synchronize()
    saved_e = [x.cpu().clone() for x in b.errs[0][0]]
    saved_q = b.q[0][0].cpu().clone()
    del b
    c = GpuRun(wl)
    for w in range(wl.workers):
        c.errs[0][0][w].copy_(saved_e[w])
    c.q[0][0].copy_(saved_q)
    for t in range(2, 4):
        c.load_inputs(t); c.step()
    torch.cuda.synchronize()
    assert torch.equal(a.ghat[0][0], c.ghat[0][0])
    assert torch.equal(a.q[0][0], c.q[0][0])
    for w in range(wl.workers):
        assert torch.equal(a.errs[0][0][w], c.errs[0][0][w])


# ------------------------------------------------------------------ argument errors
def test_dynamic_scale_on_device_matches_oracle():
    """Per-resblock dynamic scales kept on the device: psgd_step reads s_b through
    scales_device, and psgd_scale_update (backoff 1/2, growth 2, interval 2) updates them
    from the step's counts. Two blocks, five steps; block 1 has 5 nonfinite entries at
    step 1 and block 0 one at step 3, so both blocks back off and grow. The scales used at
    steps 0..4 are 2^10, 2^10, 2^11, 2^11, 2^10 for block 0 (grown after its second finite
    step, backed off after step 3) and 2^10, 2^10, 2^9, 2^9, 2^10 for block 1 (backed off
    after step 1, grown after steps 2 and 3). Each step matches the oracle run with the
    same scales, and after each update the device scale and streak equal the oracle's
    rule bit for bit."""
    psgd = _psgd()
    wl = synth.scaler_run()
    B, W = wl.blocks, wl.workers
    g = GpuRun(wl)
    o = OracleRun(wl, range(B))
    scale = torch.full((B,), 2.0 ** 10, dtype=torch.float32, device="cuda")
    streak = torch.zeros(B, dtype=torch.int32, device="cuda")
    s_ref, k_ref = [np.float32(2.0 ** 10)] * B, [0] * B
    seen = []
    for t in range(wl.steps):
        g.load_inputs(t)
        g.load_state(o)
        g.ps.step(g.grads, g.errs, g.q, None, g.ghat, g.unc_in, g.unc_out, scales_device=scale)
        res = o.step(t, scales=s_ref)
        compare_step(g, res, o)
        seen.append([float(x) for x in s_ref])
        psgd.psgd_scale_update(B, W, g.ps.counts.data_ptr(), scale.data_ptr(), streak.data_ptr(),
                               0.5, 2.0, 2, torch.cuda.current_stream().cuda_stream)
        for b in range(B):
            s_ref[b], k_ref[b] = oracle.scale_update(s_ref[b], k_ref[b], res[b].counts, 0.5, 2.0, 2)
        torch.cuda.synchronize()
        assert scale.cpu().numpy().tolist() == [float(x) for x in s_ref], t
        assert streak.cpu().numpy().tolist() == k_ref, t
    assert seen == [[2.0 ** 10, 2.0 ** 10], [2.0 ** 10, 2.0 ** 10], [2.0 ** 11, 2.0 ** 9],
                    [2.0 ** 11, 2.0 ** 9], [2.0 ** 10, 2.0 ** 10]]


def test_host_scale_below_one_matches_oracle():
    """Host scales below 1 are accepted, as device scales are: s_b = 2^-1 multiplies the
    raw gradient by 2 on unscaling (small ragged shapes, fp16, two steps)."""
    from dataclasses import replace
    wl = replace(synth.with_shapes(synth.resblock_shard(steps=2, workers=2, rank=8),
                                   ((200, 136), (72, 64))), scale_log2=-1, sigma_raw=2.0 ** -6)
    run_parity(wl)


def test_scale_update_keeps_scales_in_the_normal_range():
    """psgd_scale_update on the device at the ends of fp32's range: a growth from 2^127 and
    a backoff from 2^-126 keep S (the oracle's reading), one step inside moves it."""
    psgd = _psgd()
    scale = torch.tensor([2.0 ** 127, 2.0 ** -126, 2.0 ** 126, 2.0 ** -125], device="cuda")
    streak = torch.tensor([3, 0, 3, 0], dtype=torch.int32, device="cuda")
    counts = torch.tensor([0, 4, 0, 1], dtype=torch.int64, device="cuda")
    psgd.psgd_scale_update(4, 1, counts.data_ptr(), scale.data_ptr(), streak.data_ptr(), 0.5, 2.0,
                           4, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    want = [oracle.scale_update(s0, k0, [c], 0.5, 2.0, 4)
            for s0, k0, c in zip([2.0 ** 127, 2.0 ** -126, 2.0 ** 126, 2.0 ** -125], [3, 0, 3, 0], [0, 4, 0, 1])]
    assert scale.cpu().tolist() == [float(w[0]) for w in want]
    assert streak.cpu().tolist() == [w[1] for w in want]


def test_argument_errors_return_status():
    psgd = _psgd()
    ps = psgd.PowerSGD([(64, 32)], 1, 1, 2, "f16")
    g = torch.zeros((64, 32), dtype=torch.float16, device="cuda")
    e = torch.zeros_like(g)
    q = torch.zeros((32, 2), device="cuda")
    gh = torch.zeros((64, 32), device="cuda")
    for bad in (0.0, -1.0, float("nan")):
        with pytest.raises(psgd.PSGDError) as ex:
            ps.step([[[g]]], [[[e]]], [[q]], [bad], [[gh]])
        assert ex.value.status == psgd.PSGD_EINVAL
    with pytest.raises(psgd.PSGDError) as ex:
        ps.step([[[g]]], [[[e]]], [[q]], [float("inf")], [[gh]])
    assert ex.value.status == psgd.PSGD_EINVAL
    big = torch.zeros(64 * 32 + 8, dtype=torch.float16, device="cuda")
    mis = big[1:1 + 64 * 32].view(64, 32)  # 2-byte offset: not 16-byte aligned
    with pytest.raises(psgd.PSGDError) as ex:
        ps.step([[[mis]]], [[[e]]], [[q]], [1.0], [[gh]])
    assert ex.value.status == psgd.PSGD_EINVAL
    with pytest.raises(psgd.PSGDError) as ex:  # neither host nor device scales
        ps.step([[[g]]], [[[e]]], [[q]], None, [[gh]])
    assert ex.value.status == psgd.PSGD_EINVAL
    sd = torch.ones(2, device="cuda")
    with pytest.raises(psgd.PSGDError) as ex:  # device scales not 4-byte aligned
        ps.step([[[g]]], [[[e]]], [[q]], None, [[gh]], scales_device=sd.view(torch.uint8)[1:5])
    assert ex.value.status == psgd.PSGD_EINVAL
    ps.step([[[g]]], [[[e]]], [[q]], [1.0], [[gh]])
    ps.check()
    with pytest.raises(psgd.PSGDError) as ex:
        psgd.PowerSGD([(64, 32)], 1, 1, 40, "f16")
    assert ex.value.status == psgd.PSGD_EINVAL


def test_clip_adam_matches_oracle():
    """Global-norm clipping + Adam (fp32 moments) against the oracle, three steps. Five
    tensors span one to three 8192-element chunks (one has 3 elements); block 1 is
    skipped, and the last tensor belongs to no block. max_norm is half the gradient norm,
    so clipping is active. Each step starts both sides from the same fp32 state."""
    psgd = _psgd()
    from oracle import optim
    rng = np.random.default_rng(21)
    numel = [10000, 8192, 3, 20000, 257]
    block = [0, 0, 1, 1, -1]
    dev = "cuda"
    th = [torch.from_numpy(rng.standard_normal(n).astype(np.float32)).to(dev) for n in numel]
    m = [torch.zeros(n, device=dev) for n in numel]
    v = [torch.zeros(n, device=dev) for n in numel]
    skip = torch.tensor([0, 1], dtype=torch.uint8, device=dev)
    ws_bytes = psgd.psgd_clip_adam_workspace_size(numel)
    ws = torch.empty(ws_bytes + 256, dtype=torch.uint8, device=dev)
    ws_ptr = (ws.data_ptr() + 255) // 256 * 256
    norm_out = torch.zeros(1, device=dev)
    for step in (1, 2, 3):
        g = [torch.from_numpy((rng.standard_normal(n) * 10.0 ** -step).astype(np.float32)).to(dev)
             for n in numel]
        g64 = [x.double().cpu().numpy() for x in g]
        nrm = optim.global_norm(g64)
        c = optim.clip_coefficient(nrm, 0.5 * nrm)
        ref = [optim.adam_step(th[t].cpu().numpy(), m[t].cpu().numpy(), v[t].cpu().numpy(), g64[t],
                               step, 1e-2, 0.9, 0.99, 1e-8, clip=c,
                               skip=block[t] >= 0 and bool(skip[block[t]]))
               for t in range(len(numel))]
        th_old = [x.double().cpu().numpy() for x in th]
        psgd.psgd_clip_adam([x.data_ptr() for x in g], [x.data_ptr() for x in th],
                            [x.data_ptr() for x in m], [x.data_ptr() for x in v], numel, ws_ptr,
                            ws_bytes, torch.cuda.current_stream().cuda_stream, lr=1e-2, beta1=0.9,
                            beta2=0.99, eps=1e-8, step=step, max_norm=0.5 * nrm, block=block,
                            skip_ptr=skip.data_ptr(), num_blocks=2, norm_out_ptr=norm_out.data_ptr())
        torch.cuda.synchronize()
        assert abs(float(norm_out[0]) - nrm) <= 1e-6 * nrm
        for t in range(len(numel)):
            if block[t] >= 0 and skip[block[t]]:
                assert np.array_equal(th[t].cpu().numpy(), ref[t][0].astype(np.float32))
                continue
            d_gpu = th[t].double().cpu().numpy() - th_old[t]
            d_ref = ref[t][0] - th_old[t]
            assert rel_err(d_gpu, d_ref) <= 1e-4, (step, t)
            assert rel_err(m[t].double().cpu().numpy(), ref[t][1]) <= 1e-5, (step, t)
            assert rel_err(v[t].double().cpu().numpy(), ref[t][2]) <= 1e-5, (step, t)


# ------------------------------------------------------- vocabulary-scale uncompressed reduce
@pytest.mark.parametrize("scale_log2,length", [(10, synth.IMAGE_VOCAB * synth.D_MODEL), (0, 4099)])
def test_reduce_uncompressed_vocabulary_scale(scale_log2, length):
    """The image-token embedding gradient (8192 x 3968 fp32, 130 MB per worker) over W = 8
    workers, reduced in fp32 without compression, and a short ragged length. 0.1% of the
    entries are +-Inf/NaN. Counts are bit-exact; the mean is within 1e-4 of the oracle's
    (its fp64 mean rounded to fp32). With the skip flag set, the output is 0 and the
    counts are still reported."""
    psgd = _psgd()
    W = 8
    rows = synth.IMAGE_VOCAB if length == synth.IMAGE_VOCAB * synth.D_MODEL else 1
    cols = length // rows
    host = [synth.embedding_grad(0, w, rows=rows, cols=cols, scale_log2=scale_log2) for w in range(W)]
    dev = [h.cuda() for h in host]
    out = torch.empty(length, device="cuda")
    counts = torch.zeros(W, dtype=torch.int64, device="cuda")
    s = 2.0 ** scale_log2
    stream = torch.cuda.current_stream().cuda_stream
    psgd.psgd_reduce_uncompressed([t.data_ptr() for t in dev], length, s, out.data_ptr(),
                                  counts.data_ptr(), 0, stream)
    torch.cuda.synchronize()
    mean, _, cnt = oracle.uncompressed_mean([h.double().numpy() for h in host], s)
    assert counts.cpu().tolist() == cnt
    ref = oracle.round_to_format(mean, "f32")
    assert rel_err(f64(out), ref) <= TOL
    skip = torch.ones(1, dtype=torch.uint8, device="cuda")
    psgd.psgd_reduce_uncompressed([t.data_ptr() for t in dev], length, s, out.data_ptr(),
                                  counts.data_ptr(), skip.data_ptr(), stream)
    torch.cuda.synchronize()
    assert counts.cpu().tolist() == cnt
    assert not bool(out.any())


def test_expired_wait_reports_timeout_and_next_step_is_correct():
    """The bounded-wait path on the GPU, without a fault: with PSGD_FLAG_DEBUG_EXPIRE_WAIT
    every CTA of the decompression kernel waits on a barrier that nothing completes. The
    wait expires after its short limit, the CTA winds down (its own loads and MMAs drained,
    TMEM released), and psgd_check reports PSGD_ETIMEOUT once. A normal handle in the same
    context then runs a step that matches the oracle."""
    psgd = _psgd()
    wl = synth.with_shapes(synth.resblock_shard(steps=1, workers=2, rank=16), ((384, 256), (256, 136)))
    o = OracleRun(wl, range(wl.blocks))
    bad = GpuRun(wl, flags=psgd.PSGD_FLAG_DEBUG_EXPIRE_WAIT)
    assert bad.ps.engine == "tcgen05"
    bad.load_inputs(0)
    bad.load_state(o)
    bad.step()
    with pytest.raises(psgd.PSGDError) as ex:
        bad.ps.check()
    assert ex.value.status == psgd.PSGD_ETIMEOUT
    bad.ps.check()  # the error word was cleared
    g = GpuRun(wl)
    g.load_inputs(0)
    g.load_state(o)
    g.step()
    torch.cuda.synchronize()
    compare_step(g, o.step(0), o)
    g.ps.check()
