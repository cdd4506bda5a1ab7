"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test ties one oracle function to the pages' printed values, to a closed form, to
brute force over every bit pattern, or to a library routine on a special case. The
choice is such that a plausible mistake (a dropped term, a wrong sign or index, a
transposed operand) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import numerics as nx
from oracle import optim
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "amp_fp16_bf16_values.txt")


def _golden_sections():
    sec, out = None, {}
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("["):
                sec = line.strip("[]")
                out[sec] = []
                continue
            out[sec].append(line.split())
    return out


def _sig(x, digits):
    return float(f"{x:.{digits - 1}e}")


# ----------------------------------------------------------------- storage rounding
def test_printed_format_table():
    """§3.1 format table: min normal, max finite and epsilon at 1, as printed."""
    g = _golden_sections()
    for name, mn, mx, eps in g["formats"]:
        assert _sig(nx.min_normal(name), 5) == float(mn)
        assert _sig(nx.max_finite(name), 5) == float(mx)
        p = nx.FORMATS[name][0]
        assert _sig(2.0 ** (1 - p), 5) == float(eps)
        # epsilon at 1 is the gap to the next representable value
        assert nx.round_to_format(1.0 + 2.0 ** (1 - p), name)[()] == 1.0 + 2.0 ** (1 - p)
    for name, v in g["subnormal"]:
        assert _sig(nx.min_subnormal(name), 5) == float(v)


def test_printed_conversions():
    """§04: 1.0001 -> 1 | 1, 1e-05 -> 1.00136e-05 | 1.00136e-05, 100000 -> inf | 99840."""
    for v, f16, bf16 in _golden_sections()["convert"]:
        a = nx.round_to_format(float(v), "f16")[()]
        b = nx.round_to_format(float(v), "bf16")[()]
        assert (math.isinf(a) and f16 == "inf") or float(f"{a:g}") == float(f16)
        assert float(f"{b:g}") == float(bf16)


def test_printed_loss_scaling_table():
    """§04 / §3.2: 1e-8 is lost when written to FP16 directly, and kept by scaling it
    by 1024 before the write and dividing after."""
    for g, direct, rescued in _golden_sections()["loss_scaling"]:
        g = float(g)
        d = nx.round_to_format(g, "f16")[()]
        r = nx.round_to_format(g * 1024.0, "f16")[()] / 1024.0
        assert _sig(d, 4) == float(direct)
        assert _sig(r, 4) == float(rescued)


def test_underflow_threshold():
    """§01: |g| <= 2^-25 rounds to 0 in FP16 (a tie at 2^-25 goes to even, i.e. 0)."""
    (_, v), = _golden_sections()["underflow"]
    assert float(v) == 2.0 ** -25
    assert nx.round_to_format(2.0 ** -25, "f16")[()] == 0.0
    assert nx.round_to_format(np.nextafter(2.0 ** -25, 1.0), "f16")[()] == 2.0 ** -24


@pytest.mark.parametrize("fmt,tdt", [("f16", torch.float16), ("bf16", torch.bfloat16)])
def test_every_16bit_pattern_decodes_like_the_library(fmt, tdt):
    """Brute force: all 65,536 patterns. decode_bits (from the field definitions) must
    equal the library's reinterpretation, and every value must be a fixed point of
    round_to_format."""
    bits = np.arange(1 << 16, dtype=np.uint64)
    mine = nx.decode_bits(bits, fmt)
    lib = torch.from_numpy(bits.astype(np.int32).astype(np.int16)).view(tdt).to(torch.float64).numpy()
    same = (mine == lib) | (np.isnan(mine) & np.isnan(lib))
    assert same.all()
    assert np.array_equal(np.signbit(mine[~np.isnan(mine)]), np.signbit(lib[~np.isnan(lib)]))
    fin = np.isfinite(mine)
    assert np.array_equal(nx.round_to_format(mine[fin], fmt), mine[fin])


def test_rounding_matches_library_on_random_and_midpoints():
    """Special case that reduces to a library routine: numpy's double-to-half and
    torch's float-to-bfloat16 conversions are correctly rounded. The inputs include
    exact midpoints and their neighbours, where a wrong tie rule or a double rounding
    would show."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal(200_000) * 2.0 ** rng.integers(-30, 17, 200_000)
    h = nx.decode_bits(np.arange(0, 0x7C00, dtype=np.uint64), "f16")
    mids = (h[:-1] + h[1:]) / 2
    x = np.concatenate([x, mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 1),
                        [65504.0, 65520.0, 65519.99, 1e9, -1e9]])
    mine = nx.round_to_format(x, "f16")
    with np.errstate(over="ignore"):
        lib = x.astype(np.float16).astype(np.float64)
    assert np.array_equal(mine, lib)
    x32 = x.astype(np.float32)
    b = nx.decode_bits(np.arange(0, 0x7F80, dtype=np.uint64), "bf16")
    bm = ((b[:-1] + b[1:]) / 2).astype(np.float32)
    x32 = np.concatenate([x32, bm, -bm])
    mine_b = nx.round_to_format(x32.astype(np.float64), "bf16")
    lib_b = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(mine_b, lib_b)
    mine_f = nx.round_to_format(x, "f32")
    assert np.array_equal(mine_f, x.astype(np.float32).astype(np.float64))


# ------------------------------------------------------------- unscale / mask / count
@pytest.mark.parametrize("scale", [1.0, 2.0 ** 10, 2.0 ** -3])
def test_mask_bruteforce_all_fp16_patterns(scale):
    """Every fp16 bit pattern goes through unscale and mask. The nonfinite patterns
    are exactly those with an all-ones exponent: 2 x 2^10 = 2048 (two infinities and
    2046 NaNs). Every finite value divides exactly and is kept."""
    v = nx.decode_bits(np.arange(1 << 16, dtype=np.uint64), "f16")
    g, mask = oracle.unscale_and_mask(v, scale)
    assert int(mask.sum()) == 2048
    assert np.array_equal(mask, ~np.isfinite(v))
    assert np.all(g[mask] == 0.0)
    assert np.array_equal(g[~mask] * scale, v[~mask])


def test_accumulate_error_is_single_rounding_of_exact_sum():
    """M = RNE_E(g + E). fp16 pairs whose exact sum needs more than 24 bits are
    compared with the library rounding of their exact fp64 sum, in the cases where
    fp64 holds the sum exactly (exponent gap < 40)."""
    rng = np.random.default_rng(7)
    a = nx.decode_bits(rng.integers(0, 0x7C00, 500_000, dtype=np.uint64), "f16") * np.where(rng.random(500_000) < .5, -1, 1)
    b = nx.decode_bits(rng.integers(0, 0x7C00, 500_000, dtype=np.uint64), "f16") * np.where(rng.random(500_000) < .5, -1, 1)
    g = a / 2.0 ** 10  # unscaled gradient
    m = oracle.accumulate_error(g, b, "f16")
    assert np.array_equal(m, (g + b).astype(np.float16).astype(np.float64))
    mb = oracle.accumulate_error(g, b, "bf16")
    assert np.array_equal(mb, nx.round_to_format(g + b, "bf16"))
    # an exact midpoint sum rounds to even; one ulp away it does not
    one = oracle.accumulate_error(np.array([2.0 ** -11]), np.array([1.0]), "f16")[0]
    assert one == 1.0
    up = oracle.accumulate_error(np.array([2.0 ** -11 + 2.0 ** -40]), np.array([1.0]), "f16")[0]
    assert up == 1.0 + 2.0 ** -10


def test_skip_threshold_and_decision():
    assert oracle.skip_threshold(1.0, 8, 100) == 800
    assert oracle.skip_threshold(0.5, 3, 7) == 11  # ceil(10.5)
    assert oracle.skip_block([400, 400], 800)
    assert not oracle.skip_block([400, 399], 800)


def test_uncompressed_mean_worked_example():
    """u0 = [2, inf, -4], u1 = [4, 6, nan], s = 2 give g0 = [1, 0, -2] and
    g1 = [2, 3, 0], so the mean is [1.5, 1.5, -1] and the counts are [1, 1]."""
    mean, masks, counts = oracle.uncompressed_mean(
        [np.array([2.0, np.inf, -4.0]), np.array([4.0, 6.0, np.nan])], 2.0)
    assert np.array_equal(mean, [1.5, 1.5, -1.0])
    assert counts == [1, 1]


# --------------------------------------------------------------------- power step
def test_power_step_hand_worked_single_worker():
    """M = [[3,1],[4,2]], Q = [1,0]^T, r = 1 (worked by hand):
    P = (3,4), P-hat = (0.6,0.8), Q' = M^T P-hat = (5, 2.2), G-hat = P-hat Q'^T =
    [[3,1.32],[4,1.76]], E = M - G-hat = [[0,-0.32],[0,0.24]]."""
    m = np.array([[3.0, 1.0], [4.0, 2.0]])
    res = oracle.power_step([m], np.array([[1.0], [0.0]]))
    s = np.sign(res.p_hat[0, 0])
    assert np.allclose(s * res.p_hat[:, 0], [0.6, 0.8], atol=1e-15)
    assert np.allclose(s * res.q[:, 0], [5.0, 2.2], atol=1e-6)  # Q is stored in fp32
    assert np.allclose(res.g_hat, [[3.0, 1.32], [4.0, 1.76]], atol=1e-6)
    e, pre = oracle.error_update(m, res.g_hat, "f64")
    assert np.allclose(pre, [[0.0, -0.32], [0.0, 0.24]], atol=1e-6)


def test_power_step_hand_worked_two_workers():
    """M_0 = [[3,1],[4,2]] and M_1 = [[1,1],[0,0]] give M-bar = [[2,1],[2,1]] (rank 1).
    With Q = [1,0]^T, P = (2,2), P-hat = (1,1)/sqrt2, Q' = (2 sqrt2, sqrt2) and
    G-hat = M-bar. So E_0 = [[1,0],[2,1]], E_1 = -E_0, and the mean of E is 0."""
    m0 = np.array([[3.0, 1.0], [4.0, 2.0]])
    m1 = np.array([[1.0, 1.0], [0.0, 0.0]])
    res = oracle.power_step([m0, m1], np.array([[1.0], [0.0]]))
    assert np.allclose(res.p, [[2.0], [2.0]], atol=0)
    assert np.allclose(res.g_hat, [[2.0, 1.0], [2.0, 1.0]], atol=1e-6)
    e0, _ = oracle.error_update(m0, res.g_hat, "f64")
    e1, _ = oracle.error_update(m1, res.g_hat, "f64")
    assert np.allclose(e0, [[1.0, 0.0], [2.0, 1.0]], atol=1e-6)
    assert np.allclose(e0 + e1, 0.0, atol=1e-6)


def test_exact_reconstruction_of_planted_low_rank():
    """rank(M) <= r and a generic Q give span(MQ) = col(M), so G-hat = M. The planted
    U V^T (rank 3, r = 4) of the small fp32 workload must come back within 1e-12."""
    wl = synth.planted_rank3()
    g = synth.grad(wl, 0, 0, 0, 0).double().numpy()
    assert np.linalg.matrix_rank(g) == 3
    q = synth.q0(wl, 0, 0).double().numpy()
    res = oracle.power_step([g, g], q)
    proj = res.p_hat @ (res.p_hat.T @ g)
    assert np.linalg.norm(proj - g) / np.linalg.norm(g) <= 1e-12
    # G-hat also carries the fp32 storage of Q: ||dQ|| <= 2^-24 ||Q|| = 2^-24 ||G-hat||
    assert np.linalg.norm(res.g_hat - g) / np.linalg.norm(g) <= 2.0 ** -24


def test_full_rank_identity_case():
    """W = 1 and r = min(m, n): span(P) is the whole column space, so G-hat = M."""
    rng = np.random.default_rng(3)
    m = rng.standard_normal((20, 12))
    res = oracle.power_step([m], rng.standard_normal((12, 12)))
    assert np.linalg.norm(res.p_hat @ (res.p_hat.T @ m) - m) / np.linalg.norm(m) <= 1e-12
    assert np.linalg.norm(res.g_hat - m) / np.linalg.norm(m) <= 2.0 ** -24


def test_zero_input_gives_zero():
    z = np.zeros((16, 8))
    res = oracle.power_step([z, z], np.ones((8, 2)))
    assert np.all(res.g_hat == 0) and np.all(res.q == 0)


def test_orthonormality():
    rng = np.random.default_rng(4)
    ms = [rng.standard_normal((300, 90)) for _ in range(3)]
    res = oracle.power_step(ms, rng.standard_normal((90, 17)))
    assert np.abs(res.p_hat.T @ res.p_hat - np.eye(17)).max() <= 1e-12
    # span(P-hat) = span(P): projecting P onto P-hat leaves nothing
    assert np.linalg.norm(res.p - res.p_hat @ (res.p_hat.T @ res.p)) <= 1e-12 * np.linalg.norm(res.p)


def test_worker_mean_equals_power_step_on_mean():
    """P and Q depend on the workers only through M-bar, because the mean is linear.
    The W-worker step must equal a one-worker step on M-bar. This mirrors the
    sharded-vs-full equivalence check in "AIGC 基本功|数据并行与 ZeRO 显存切分", §4.2."""
    rng = np.random.default_rng(5)
    ms = [rng.standard_normal((120, 70)) for _ in range(4)]
    q = rng.standard_normal((70, 6))
    a = oracle.power_step(ms, q)
    b = oracle.power_step([sum(ms) / 4], q)
    mbar = sum(ms) / 4
    pa = a.p_hat @ (a.p_hat.T @ mbar)
    pb = b.p_hat @ (b.p_hat.T @ mbar)
    assert np.abs(pa - pb).max() <= 1e-12 * np.abs(pa).max()
    assert np.abs(a.p - b.p).max() <= 1e-12 * np.abs(a.p).max()
    # the stored Q differs at most by its fp32 rounding
    assert np.linalg.norm(a.g_hat - b.g_hat) <= 2.0 ** -23 * np.linalg.norm(a.g_hat)


def test_basis_invariance_householder_vs_mgs2():
    """G-hat = P-hat P-hat^T M-bar depends only on span(P), and a rotation of P-hat
    carries through the next Q. So a trajectory of several steps with error feedback
    is the same with Householder QR and with Gram-Schmidt."""
    rng = np.random.default_rng(6)
    m_, n_, r, W = 90, 60, 5, 3
    q = rng.standard_normal((n_, r))
    sa = oracle.BlockState(e=[[np.zeros((m_, n_)) for _ in range(W)]], q=[q.copy()])
    sb = oracle.BlockState(e=[[np.zeros((m_, n_)) for _ in range(W)]], q=[q.copy()])
    for t in range(4):
        grads = [[rng.standard_normal((m_, n_)) for _ in range(W)]]
        ra = oracle.block_step(grads, sa, 1.0, "f64", orth="householder")
        rb = oracle.block_step(grads, sb, 1.0, "f64", orth="mgs2")
        scale = np.abs(ra.g_hat[0]).max()
        assert np.abs(ra.g_hat[0] - rb.g_hat[0]).max() <= 1e-11 * scale
        for w in range(W):
            assert np.abs(sa.e[0][w] - sb.e[0][w]).max() <= 1e-11 * scale


def test_error_feedback_identity():
    """M_w = G-hat + E_w before rounding, and the stored E_w is the RNE of that value
    (within half an ulp of E's type). The residual mean is orthogonal to P-hat, up to
    the fp32 rounding of Q."""
    wl = synth.resblock_shard(steps=1, shapes=((200, 136),), workers=3, rank=7)
    st = oracle.BlockState(e=[[np.zeros((200, 136)) for _ in range(3)]],
                           q=[synth.q0(wl, 0, 0).double().numpy()])
    grads = [[synth.grad(wl, 0, 0, 0, w).double().numpy() for w in range(3)]]
    res = oracle.block_step(grads, st, wl.scale(0), "f16")
    for w in range(3):
        assert np.array_equal(res.m[0][w], res.g_hat[0] + res.e_pre[0][w]) or \
            np.abs(res.m[0][w] - res.g_hat[0] - res.e_pre[0][w]).max() <= 1e-18
        assert np.array_equal(st.e[0][w], nx.round_to_format(res.e_pre[0][w], "f16"))
    mean_pre = sum(res.e_pre[0]) / 3
    ortho = res.p_hat[0].T @ mean_pre
    assert np.abs(ortho).max() <= 1e-6 * np.abs(res.p_hat[0].T @ (sum(res.m[0]) / 3)).max()


def test_eckart_young_bound_and_convergence():
    """Without error feedback, repeated warm-started steps on a fixed M = U diag(1/k) V^T
    are subspace iteration. ||M - G-hat|| never falls below sqrt(sum_{k>r} sigma_k^2),
    the Eckart-Young bound, and it converges to it."""
    rng = np.random.default_rng(8)
    m_, n_, r = 64, 48, 4
    u, _ = np.linalg.qr(rng.standard_normal((m_, n_)))
    v, _ = np.linalg.qr(rng.standard_normal((n_, n_)))
    sig = 1.0 / np.arange(1, n_ + 1)
    mm = (u * sig) @ v.T
    bound = math.sqrt(float(np.sum(sig[r:] ** 2)))
    q = rng.standard_normal((n_, r))
    errs = []
    for _ in range(60):
        res = oracle.power_step([mm, mm], q)
        q = res.q
        errs.append(np.linalg.norm(mm - res.g_hat))
    assert min(errs) >= bound * (1 - 1e-7)
    assert errs[-1] <= bound * (1 + 1e-6)
    assert errs[0] > errs[-1]


def test_skip_keeps_state_and_zeroes_output():
    """A block whose every entry is nonfinite on every worker is skipped. E and Q are
    unchanged, G-hat and the gains/biases are 0, and the counts are reported."""
    rng = np.random.default_rng(9)
    e0 = [[rng.standard_normal((8, 6)) for _ in range(2)]]
    q = rng.standard_normal((6, 2))
    st = oracle.BlockState(e=[[x.copy() for x in e0[0]]], q=[q.copy()])
    grads = [[np.full((8, 6), np.nan), np.full((8, 6), np.inf)]]
    unc = [np.full(4, np.inf), np.full(4, -np.inf)]
    res = oracle.block_step(grads, st, 4.0, "f64", unc=unc)
    assert res.skip and res.counts == [52, 52]
    assert all(np.array_equal(st.e[0][w], e0[0][w]) for w in range(2))
    assert np.array_equal(st.q[0], q)
    assert np.all(res.g_hat[0] == 0) and np.all(res.unc_out == 0)
    # one finite entry anywhere in the block defeats the skip at T = 1
    grads[0][1][3, 2] = 1.0
    res2 = oracle.block_step(grads, st, 4.0, "f64", unc=unc)
    assert not res2.skip and res2.counts == [52, 51]


def test_partial_nonfinite_is_zeroed_and_counted():
    wl = synth.stress(steps=1, shapes=((64, 40),), blocks=1, workers=2, rank=3, frac=0.05)
    g = synth.grad(wl, 0, 0, 0, 0).double().numpy()
    want = int(round(0.05 * 64 * 40))
    gg, mask = oracle.unscale_and_mask(g, wl.scale(0))
    assert int(mask.sum()) == want
    assert np.all(np.isfinite(gg))


# --------------------------------------------------------------------- accounting
def test_compression_ratio_matches_pages():
    """[card] 方法适配 / 证据: total rank 896, which is 112 per GPU's shard, and about
    86% compression. [notes]: 85%. For the four 1/8-column shard matrices at r = 112
    the factors are 3,610,880 of 23,617,536 entries, i.e. 84.7% compression."""
    shapes = synth.SHARD_SHAPES
    frac = oracle.compressed_fraction(shapes, 112)
    assert sum((m + n) * 112 for m, n in shapes) == 3_610_880
    assert sum(m * n for m, n in shapes) == 23_617_536
    assert 0.84 <= 1 - frac <= 0.87
    assert round(100 * (1 - frac)) == 85
    # rank 896 on the unsharded matrices would give only ~70%: the per-shard reading
    full = ((3968, 3 * 3968), (3968, 3968), (3968, 4 * 3968), (4 * 3968, 3968))
    assert 1 - oracle.compressed_fraction(full, 896) < 0.71


def test_parameter_count_is_12B():
    """64 layers of 12 d_model^2 weights with d_model = 3968 is 12.09e9 parameters, the
    "12B" of the pages ([card] 计算设置)."""
    assert 64 * 12 * 3968 ** 2 == 12_092_178_432
    assert 64 * sum(m * n for m, n in synth.SHARD_SHAPES) * 8 == 64 * 12 * 3968 ** 2


# ------------------------------------------------------------- dynamic scale ([amp] §3.2)
def _run_scaler(s0, events, backoff, growth, interval):
    s, k, trace = s0, 0, []
    for nonfinite in events:
        s, k = oracle.scale_update(s, k, [0, 1] if nonfinite else [0, 0], backoff, growth,
                                   interval)
        trace.append((float(s), k))
    return trace


def test_scale_update_hand_worked_sequence_drops_below_one():
    """S0 = 1, backoff 1/2, growth 2, interval 2, events N F F N N F (N: the block held an
    Inf/NaN). By the rule: 1/2 (streak 0), 1/2 (1), 1 (grown, 0), 1/2, 1/4, 1/4 (1). The
    scale goes below 1, which the page says can happen."""
    assert _run_scaler(1.0, [1, 0, 0, 1, 1, 0], 0.5, 2.0, 2) == [
        (0.5, 0), (0.5, 1), (1.0, 0), (0.5, 0), (0.25, 0), (0.25, 1)]


def test_scale_update_counts_any_worker():
    """One nonfinite entry on any worker backs the block off; zero counts everywhere do
    not."""
    assert oracle.scale_update(8.0, 3, [0, 0, 0, 1], 0.5, 2.0, 100) == (4.0, 0)
    assert oracle.scale_update(8.0, 3, [0, 0, 0, 0], 0.5, 2.0, 100) == (8.0, 4)


def test_scale_update_closed_form_over_random_events():
    """With power-of-two factors every product is exact, so after any event sequence
    S = 2^(e0 + growths - backoffs). The counts come from a run-length reading of the
    sequence, not from the update: every event N is one backoff; a run of L finite
    events after a reset gives floor(L / K) growths and leaves L mod K in the streak."""
    rng = np.random.default_rng(11)
    events = (rng.random(600) < 0.25).astype(int)
    K = 3
    trace = _run_scaler(2.0 ** 5, events, 0.5, 2.0, K)
    backoffs = int(events.sum())
    runs, cur = [], 0
    for ev in events:
        if ev:
            runs.append(cur)
            cur = 0
        else:
            cur += 1
    runs.append(cur)
    growths = sum(L // K for L in runs)
    e = 5 + growths - backoffs
    assert -120 < e < 120  # stays in fp32's normal range for this seed
    assert trace[-1] == (2.0 ** e, runs[-1] % K)


def test_scale_update_rounds_each_product_to_fp32():
    """Backoff 0.3 is not a power of two. fp32(0.3) = 0.300000011920928955078125, so
    1000 * fp32(0.3) = 300.0000119209..., which is within half an fp32 ulp (2^-16 at 300)
    of 300: S' = 300 exactly. A second backoff: 300 * fp32(0.3) = 90.0000035762...,
    which rounds to 90 (half an ulp there is 2^-18 = 3.8e-6)."""
    s, _ = oracle.scale_update(1000.0, 0, [1], 0.3, 2.0, 4)
    assert s == np.float32(300.0) and s.dtype == np.float32
    s, _ = oracle.scale_update(s, 0, [1], 0.3, 2.0, 4)
    assert s == np.float32(90.0)


def test_scale_update_stays_a_finite_normal_float():
    """At the ends of fp32's range the update keeps S: 2^127 * 2 overflows and 2^-126 / 2
    is subnormal, so both stay; the streak still restarts. One step inside the range
    moves as usual (2^126 * 2 = 2^127, 2^-125 / 2 = 2^-126)."""
    big, tiny = np.float32(2.0 ** 127), np.float32(2.0 ** -126)
    assert oracle.scale_update(big, 3, [0], 0.5, 2.0, 4) == (big, 0)
    assert oracle.scale_update(tiny, 2, [5], 0.5, 2.0, 4) == (tiny, 0)
    assert oracle.scale_update(np.float32(2.0 ** 126), 3, [0], 0.5, 2.0, 4)[0] == big
    assert oracle.scale_update(np.float32(2.0 ** -125), 0, [1], 0.5, 2.0, 4)[0] == tiny
    # a backoff that would go below the normal range from a non-power-of-two scale
    s = np.float32(1.5 * 2.0 ** -126)
    assert oracle.scale_update(s, 0, [1], 0.5, 2.0, 4)[0] == s


# ------------------------------------------- consumer of G-hat: clipping + Adam ([amp] §6.2)


def test_global_norm_is_the_norm_of_the_concatenated_shards():
    """[amp] §6.2: the global norm is the root of the all-reduced local sums of squares.
    It equals the 2-norm of all shards laid end to end (numpy's own norm)."""
    rng = np.random.default_rng(5)
    shards = [rng.standard_normal(s) for s in ((7, 3), (11,), (2, 5, 4))]
    flat = np.concatenate([x.reshape(-1) for x in shards])
    assert math.isclose(optim.global_norm(shards), float(np.linalg.norm(flat)), rel_tol=1e-14)
    assert optim.global_norm([np.zeros(3)]) == 0.0
    assert optim.global_norm([np.array([3.0]), np.array([4.0])]) == 5.0


def test_clip_coefficient_hand_worked():
    assert optim.clip_coefficient(5.0, 1.0) == 0.2
    assert optim.clip_coefficient(0.5, 1.0) == 1.0
    assert optim.clip_coefficient(1.0, 1.0) == 1.0
    assert optim.clip_coefficient(0.0, 1.0) == 1.0
    # clipping rescales the global norm to exactly C (up to rounding)
    g = [np.array([3.0, 4.0]), np.array([12.0])]
    c = optim.clip_coefficient(optim.global_norm(g), 2.0)
    assert math.isclose(optim.global_norm([x * c for x in g]), 2.0, rel_tol=1e-15)


def test_adam_first_step_closed_form():
    """From zero moments, bias correction makes m_hat = g and v_hat = g^2, so the first
    step moves theta by exactly -lr g / (|g| + eps)."""
    g = np.array([0.5, -2.0, 1e-3, 0.0])
    th, m, v = optim.adam_step(np.ones(4), np.zeros(4), np.zeros(4), g, 1, 1e-2, 0.9, 0.999, 1e-8)
    assert np.allclose(th, 1.0 - 1e-2 * g / (np.abs(g) + 1e-8), rtol=0, atol=1e-15)
    assert np.allclose(m, 0.1 * g) and np.allclose(v, 0.001 * g * g)


def test_adam_constant_gradient_steps_tend_to_lr():
    """For a constant gradient g, m_t = (1 - b1^t) g and v_t = (1 - b2^t) g^2 exactly, so
    every bias-corrected step is lr * g / (|g| + eps): with eps = 0 it is lr sign(g)."""
    g = np.array([2.0, -0.25])
    th, m, v = np.zeros(2), np.zeros(2), np.zeros(2)
    for t in range(1, 40):
        before = th
        th, m, v = optim.adam_step(th, m, v, g, t, 0.1, 0.9, 0.99, 0.0)
        assert np.allclose(th - before, -0.1 * np.sign(g), rtol=0, atol=1e-12), t
        assert np.allclose(m, (1 - 0.9 ** t) * g, rtol=1e-12)


def test_adam_is_invariant_to_gradient_scale_without_eps_and_skip_keeps_state():
    rng = np.random.default_rng(9)
    gs = [rng.standard_normal(6) for _ in range(5)]
    a = b = (np.zeros(6), np.zeros(6), np.zeros(6))
    for t, g in enumerate(gs, 1):
        a = optim.adam_step(*a, g, t, 1e-3, 0.9, 0.999, 0.0)
        b = optim.adam_step(*b, 1024.0 * g, t, 1e-3, 0.9, 0.999, 0.0)
    assert np.allclose(a[0], b[0], rtol=1e-12, atol=0)
    st = (np.ones(3), np.full(3, 0.5), np.full(3, 0.25))
    out = optim.adam_step(*st, np.full(3, np.nan), 3, 1e-3, 0.9, 0.999, 1e-8, skip=True)
    assert all(np.array_equal(x, y) for x, y in zip(out, st))
