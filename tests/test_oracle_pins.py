"""Pins for the CPU oracle: each test checks it against something other than
itself -- values and tolerances printed on the method's pages, closed forms,
brute force, or library routines that the method reduces to in a special case.

Sources: '[XPU] Implemented 8bit optimizers in triton #1692' (benchmark script
test_optimizer8bit), 'optim_overview.md' (bitsandbytes docs), 'Support
skip_zeros in the XPU Triton optimizer kernels #2097', '8-bit Optimizers via
Block-wise Quantization' (abstract).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


S = oracle.create_qmap(True)
U = oracle.create_qmap(False)


# ---------------------------------------------------------------------------
# the dynamic map
# ---------------------------------------------------------------------------

def byte_structure_map(signed: bool) -> np.ndarray:
    """Enumerate all 256 code bytes by their bit layout (sign bit, k zero bits
    = exponent -k, an indicator 1, then the fraction bits) -- a construction
    independent of the oracle's per-exponent loop."""
    vals = []
    for byte in range(256):
        if signed:
            sign = -1.0 if byte & 0x80 else 1.0
            rest, width = byte & 0x7F, 7
        else:
            sign, rest, width = 1.0, byte, 8
        if rest == 0:
            vals.append(1.0 if sign < 0 else 0.0)   # the "negative zero" slot holds +1.0
            continue
        if not signed and rest == 1:
            vals.append(1.0)                        # unsigned: all-zero run, no fraction
            continue
        k = width - rest.bit_length()               # leading zero bits = exponent
        fbits = rest.bit_length() - 1               # bits after the indicator
        if not signed:
            if k == width - 1:                      # handled above (rest == 1)
                raise AssertionError
        frac_index = rest & ((1 << fbits) - 1)
        level = 10.0 ** (-k) * (0.1 + (frac_index + 0.5) * 0.9 / (1 << fbits))
        vals.append(sign * level)
    return np.sort(np.array(vals, dtype=np.float64)).astype(np.float32)


@pytest.mark.parametrize("signed", [True, False])
def test_qmap_matches_byte_structure_enumeration(signed):
    q = oracle.create_qmap(signed)
    np.testing.assert_array_equal(q, byte_structure_map(signed))


def test_qmap_closed_form_values():
    gold = golden("qmap_closed_form.json")
    for name, q in (("signed", oracle.create_qmap(True)), ("unsigned", oracle.create_qmap(False))):
        for idx, dec in gold[name].items():
            assert q[int(idx)] == np.float32(float(dec)), (name, idx, q[int(idx)], dec)
        # number of levels in each decade [10^-(k+1), 10^-k)
        for k, cnt in gold["levels_per_exponent"][name].items():
            k = int(k)
            lo, hi = 10.0 ** (-(k + 1)), 10.0 ** (-k)
            got = int(np.count_nonzero((q > lo) & (q < hi)))
            assert got == cnt, (name, k, got, cnt)


def test_qmap_monotone_symmetric_endpoints():
    S, U = oracle.create_qmap(True), oracle.create_qmap(False)
    for q in (S, U):
        assert q.dtype == np.float32 and q.shape == (256,)
        assert np.all(np.diff(q.astype(np.float64)) > 0)
        assert q[255] == 1.0
    assert S[127] == 0.0 and U[0] == 0.0
    assert S.min() > -1.0 and U.min() == 0.0
    for j in range(1, 128):
        assert S[127 + j] == -S[127 - j]


# ---------------------------------------------------------------------------
# storage dtypes
# ---------------------------------------------------------------------------

def _rounding_ties():
    # binary32 values exactly halfway between two bfloat16 / binary16 values,
    # with both parities of the last kept bit
    rng = np.random.default_rng(7)
    hi = rng.integers(0, 1 << 16, 4000, dtype=np.uint32)
    bf16_ties = ((hi << 16) | 0x8000).astype(np.uint32).view(np.float32)
    mant = rng.integers(0, 1 << 10, 4000, dtype=np.uint32)
    expo = rng.integers(103, 143, 4000, dtype=np.uint32)            # normal binary16 range
    f16_ties = ((expo << 23) | (mant << 13) | 0x1000).astype(np.uint32).view(np.float32)
    sub = (rng.integers(1, 1 << 10, 2000).astype(np.float32) + np.float32(0.5)) * np.float32(2.0 ** -24)
    return np.concatenate([bf16_ties, -bf16_ties, f16_ties, -f16_ties, sub, -sub])


def _edge_floats():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        _rounding_ties(),
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-6).astype(np.float32),
        (rng.standard_normal(5000) * 7e4).astype(np.float32),
        np.array([0.0, -0.0, 65504.0, 65519.0, 65520.0, 65536.0, 6e-8, 3e-8, 2.9802322e-08,
                  5.96e-8, 1e-40, -1e-40, 3.4e38, np.inf, -np.inf], dtype=np.float32),
        rng.integers(0, 2**32, 20000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    return x[np.isfinite(x) | np.isinf(x)]


def test_bf16_rounding_matches_torch():
    x = _edge_floats()
    mine = oracle.to_storage(x, "bf16")
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(mine, ref)
    back = oracle.to_f32(mine, "bf16")
    np.testing.assert_array_equal(back, torch.from_numpy(ref.view(np.int16)).view(
        torch.bfloat16).float().numpy())


def test_f16_rounding_matches_numpy():
    x = _edge_floats()
    mine = oracle.to_storage(x, "f16")
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(mine, ref)
    np.testing.assert_array_equal(oracle.to_f32(mine, "f16"), ref.view(np.float16).astype(np.float32))


# ---------------------------------------------------------------------------
# nearest-code search
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("q", [S, U], ids=["signed", "unsigned"])
def test_code_is_nearest_level_brute_force(q):
    mid = oracle.midpoints(q)
    rng = np.random.default_rng(2)
    lo = -1.0 if q[0] < 0 else 0.0
    xs = np.concatenate([rng.uniform(lo, 1.0, 3000),
                         np.sign(rng.uniform(lo, 1.0, 3000)) * 10 ** rng.uniform(-8, 0, 3000)])
    xs = xs.astype(np.float32)
    for x in xs:
        c = oracle.code(mid, x)
        d = np.abs(q.astype(np.float64) - float(x))
        best = int(np.argmin(d))
        if c != best:
            # only at an (almost) exact tie between two neighbouring levels
            assert abs(c - best) == 1
            assert abs(d[c] - d[best]) <= 2 * np.spacing(np.float32(abs(x)))


def test_code_tie_goes_to_lower_level_and_exact_levels_map_to_themselves():
    for q in (S, U):
        mid = oracle.midpoints(q)
        for i in range(255):
            assert oracle.code(mid, mid[i]) == i          # exact midpoint: lower index
            assert oracle.code(mid, np.nextafter(mid[i], np.float32(2))) == i + 1
        for c in range(256):
            assert oracle.code(mid, q[c]) == c


# ---------------------------------------------------------------------------
# block-wise quantization
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("blocksize", [256, 2048])
@pytest.mark.parametrize("scale_exp", [0, -3, 5])
def test_quantize_round_trips_every_level(blocksize, scale_exp):
    rng = np.random.default_rng(3)
    for q in (S, U):
        reps = blocksize // 256
        blocks = []
        for _ in range(3):
            blk = np.tile(q, reps)
            rng.shuffle(blk)
            blocks.append(blk)
        x = (np.concatenate(blocks) * np.float32(2.0 ** scale_exp)).astype(np.float32)
        codes, absmax = oracle.quantize_blockwise(x, "f32", q, blocksize)
        np.testing.assert_array_equal(absmax, np.float32(2.0 ** scale_exp))
        np.testing.assert_array_equal(q[codes], x / np.float32(2.0 ** scale_exp))
        back = oracle.dequantize_blockwise(codes, absmax, q, blocksize, "f32")
        np.testing.assert_array_equal(back, x)


def test_quantize_error_bound_absmax_and_ragged_tail():
    rng = np.random.default_rng(4)
    n, B = 256 * 5 + 77, 256
    for q, x in ((S, rng.standard_normal(n).astype(np.float32) * 0.01),
                 (U, np.abs(rng.standard_normal(n)).astype(np.float32) * 1e-5)):
        codes, absmax = oracle.quantize_blockwise(x, "f32", q, B)
        assert absmax.shape == (6,)
        for b in range(6):
            assert absmax[b] == np.abs(x[b * B:(b + 1) * B]).max()
        back = oracle.dequantize_blockwise(codes, absmax, q, B, "f32")
        gaps = np.diff(q.astype(np.float64))
        # |x - deq| <= absmax * (largest gap next to the chosen level) / 2, plus one rounding
        c = codes.astype(np.int64)
        local = np.maximum(gaps[np.clip(c - 1, 0, 254)], gaps[np.clip(c, 0, 254)])
        amax = np.repeat(absmax, B)[:n].astype(np.float64)
        err = np.abs(back.astype(np.float64) - x)
        assert np.all(err <= amax * (local / 2 + 2.0 ** -22))
        # the tail block quantizes like a stand-alone block
        c_tail, a_tail = oracle.quantize_blockwise(x[5 * B:], "f32", q, B)
        np.testing.assert_array_equal(c_tail, codes[5 * B:])
        assert a_tail[0] == absmax[5]


def test_quantize_zero_block_is_zero_code():
    for q, zc in ((S, 127), (U, 0)):
        codes, absmax = oracle.quantize_blockwise(np.zeros(300, np.float32), "f32", q, 256)
        assert np.all(codes == zc) and np.all(absmax == 0)
        assert q[zc] == 0.0


def test_quantize_nan_makes_its_block_absmax_nan():
    """READING (a NaN in the block): absmax is the IEEE 754-2019 maximum, NaN
    when any |x| is; the block is then normalised by 0 like an all-zero
    block (every value takes the code of 0, the NaN code 0), and the other
    blocks are as if quantized alone."""
    x = workloads.normal(600, 0.1, 3).astype(np.float32)
    x[10] = np.nan
    for q, zc in ((S, 127), (U, 0)):
        codes, absmax = oracle.quantize_blockwise(x, "f32", q, 256)
        assert np.isnan(absmax[0]) and not np.isnan(absmax[1:]).any()
        assert codes[10] == 0
        assert np.all(np.delete(codes[:256], 10) == zc)
        c2, a2 = oracle.quantize_blockwise(x[256:], "f32", q, 256)
        assert np.array_equal(codes[256:], c2) and np.array_equal(absmax[1:], a2)


def test_step_nan_state_makes_its_block_absmax_nan():
    """The same reading in the step: a NaN gradient gives a NaN first moment,
    so that block's absmax is NaN and its codes are the code of 0 (the NaN's:
    0); p takes the NaN, every other element and block steps as without it."""
    n, B = 700, 256
    g = workloads.normal(n, 1e-2, 11).astype(np.float32)
    ohp = oracle.HParams(optim="momentum", lr=0.01, beta1=0.9, step=1)
    runs = []
    for bad in (True, False):
        gg = g.copy()
        if bad:
            gg[300] = np.nan
        p = workloads.normal(n, 0.1, 12).astype(np.float32)
        t = oracle.TensorState(p, *oracle.zero_state("momentum", n, 8, B, S, None), 8)
        oracle.step(ohp, t, gg, "f32", B, S, None)
        runs.append(t)
    nan_run, ref = runs
    assert np.isnan(nan_run.absmax1[1]) and np.isnan(nan_run.p[300])
    assert nan_run.s1[300] == 0 and np.all(np.delete(nan_run.s1[256:512], 300 - 256) == 127)
    keep = np.r_[0:256, 512:n]
    assert np.array_equal(nan_run.s1[keep], ref.s1[keep])
    assert np.array_equal(nan_run.absmax1[[0, 2]], ref.absmax1[[0, 2]])
    assert np.array_equal(np.delete(nan_run.p, 300), np.delete(ref.p, 300))


def test_quantize_half_inputs_widen_exactly():
    rng = np.random.default_rng(5)
    x = rng.standard_normal(1000).astype(np.float32)
    for dt in ("bf16", "f16"):
        xs = oracle.to_storage(x, dt)
        c1, a1 = oracle.quantize_blockwise(xs, dt, S, 256)
        c2, a2 = oracle.quantize_blockwise(oracle.to_f32(xs, dt), "f32", S, 256)
        np.testing.assert_array_equal(c1, c2)
        np.testing.assert_array_equal(a1, a2)


# ---------------------------------------------------------------------------
# 32-bit-state steps against torch.optim (the comparators the benchmark
# script pairs with the 8-bit optimizers)
# ---------------------------------------------------------------------------

TORCH_CASES = {
    "adam": (lambda p, wd: torch.optim.Adam([p], lr=1e-3, betas=(0.9, 0.999), eps=1e-8,
                                            weight_decay=wd),
             dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8), ["exp_avg", "exp_avg_sq"]),
    "adamw": (lambda p, wd: torch.optim.AdamW([p], lr=1e-3, betas=(0.9, 0.999), eps=1e-8,
                                              weight_decay=wd),
              dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8), ["exp_avg", "exp_avg_sq"]),
    "momentum": (lambda p, wd: torch.optim.SGD([p], lr=0.01, momentum=0.9, weight_decay=wd),
                 dict(lr=0.01, beta1=0.9), ["momentum_buffer"]),
    "rmsprop": (lambda p, wd: torch.optim.RMSprop([p], lr=0.01, alpha=0.9, eps=1e-8,
                                                  weight_decay=wd),
                dict(lr=0.01, beta1=0.9, eps=1e-8), ["square_avg"]),
    "adagrad": (lambda p, wd: torch.optim.Adagrad([p], lr=0.01, eps=1e-8, weight_decay=wd),
                dict(lr=0.01, eps=1e-8), ["sum"]),
}


@pytest.mark.parametrize("optim", sorted(TORCH_CASES))
@pytest.mark.parametrize("wd", [0.0, 1e-2])
@pytest.mark.parametrize("gnorm_scale", [1.0, 0.5])
def test_32bit_step_matches_torch_optim(optim, wd, gnorm_scale):
    make, hpkw, names = TORCH_CASES[optim]
    n = 4099
    p0 = workloads.normal(n, 0.1, 10)
    pt = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = make(pt, wd)
    s1, s2, _, _ = oracle.zero_state(optim, n, 32, 256)
    t = oracle.TensorState(p0.copy(), s1, s2, None, None, 32)
    for k in range(1, 8):
        g = workloads.normal(n, 0.01, 100 + k)
        g[::17] = 0.0
        g[5::29] *= np.float32(1e-7)                 # sqrt(v) comparable to eps
        pt.grad = torch.from_numpy(g * np.float32(gnorm_scale))
        opt.step()
        hp = oracle.HParams(optim=optim, weight_decay=wd, step=k, gnorm_scale=gnorm_scale,
                            **hpkw)
        oracle.step(hp, t, g, "f32", 256)
        # torch may fuse p + (-lr) * x; the difference is a rounding of an lr-sized update
        np.testing.assert_allclose(t.p, pt.detach().numpy(), rtol=2e-6, atol=hp.lr * 1e-5)
        st = opt.state[pt]
        # torch rounds differently where terms nearly cancel (Adam's m is a lerp, SGD adds
        # decay and momentum in another order), so the floor is a few ulps of the largest
        # state value
        for mine, name in zip((t.s1[:n], t.s2), names):
            ref = st[name].numpy()
            np.testing.assert_allclose(mine, ref, rtol=2e-5, atol=1e-6 * np.abs(ref).max())


def test_lion_worked_example():
    ex = golden("lion_worked_example.json")
    t = oracle.TensorState(np.array([ex["p0"]], np.float32), np.zeros(1, np.float32), None, None,
                           None, 32)
    for k, g in enumerate(ex["grads"]):
        hp = oracle.HParams(optim="lion", lr=ex["lr"], beta1=ex["beta1"], beta2=ex["beta2"],
                            step=k + 1)
        oracle.step(hp, t, np.array([g], np.float32), "f32", 256)
        assert t.p[0] == np.float32(ex["p_after"][k])
        assert abs(t.s1[0] - ex["m_after"][k]) < 1e-7


def test_lion_constant_gradient_closed_form():
    # constant g: m_k = (1 - b2^k) g, c_k has the sign of g, p_k = p_{k-1}(1-lr wd) - lr sign(g)
    n, lr, wd, b2 = 1000, 1e-3, 0.1, 0.99
    g = workloads.normal(n, 1e-3, 20)
    g[g == 0] = 1e-3
    p0 = workloads.normal(n, 0.5, 21)
    t = oracle.TensorState(p0.copy(), np.zeros(n, np.float32), None, None, None, 32)
    p_ref = p0.astype(np.float64)
    for k in range(1, 21):
        hp = oracle.HParams(optim="lion", lr=lr, beta1=0.9, beta2=b2, weight_decay=wd, step=k)
        oracle.step(hp, t, g, "f32", 256)
        p_ref = p_ref * (1 - lr * wd) - lr * np.sign(g)
        np.testing.assert_allclose(t.s1, (1 - b2 ** k) * g.astype(np.float64), rtol=1e-5)
    np.testing.assert_allclose(t.p, p_ref, rtol=1e-6, atol=1e-6)


def test_ademamix_alpha_zero_is_adamw():
    n, wd = 3000, 1e-2
    p0 = workloads.normal(n, 0.1, 30)
    pt = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.AdamW([pt], lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=wd)
    s1, s2, _, _ = oracle.zero_state("ademamix", n, 32, 256)
    t = oracle.TensorState(p0.copy(), s1, s2, None, None, 32)
    for k in range(1, 8):
        g = workloads.normal(n, 0.01, 300 + k)
        pt.grad = torch.from_numpy(g.copy())
        opt.step()
        hp = oracle.HParams(optim="ademamix", lr=1e-3, beta1=0.9, beta2=0.999, beta3=0.9999,
                            alpha=0.0, eps=1e-8, weight_decay=wd, step=k)
        oracle.step(hp, t, g, "f32", 256)
        np.testing.assert_allclose(t.p, pt.detach().numpy(), rtol=2e-6, atol=1e-9)
        np.testing.assert_allclose(t.s1[:n], opt.state[pt]["exp_avg"].numpy(), rtol=2e-5,
                                   atol=1e-9)
        np.testing.assert_allclose(t.s2, opt.state[pt]["exp_avg_sq"].numpy(), rtol=2e-5,
                                   atol=1e-13)


def test_ademamix_constant_gradient_closed_form():
    # constant g, no decay, no schedule: m1/bc1 = g, nu/bc2 = g^2, m2_t = (1 - b3^t) g,
    # so p_t = p_{t-1} - lr (1 + alpha (1 - b3^t)) g / (|g| + eps)
    n, lr, alpha, b3 = 500, 1e-3, 5.0, 0.99
    g = workloads.normal(n, 1e-3, 40)
    p0 = workloads.normal(n, 0.1, 41)
    s1, s2, _, _ = oracle.zero_state("ademamix", n, 32, 256)
    t = oracle.TensorState(p0.copy(), s1, s2, None, None, 32)
    gd = g.astype(np.float64)
    p_ref = p0.astype(np.float64)
    for k in range(1, 31):
        hp = oracle.HParams(optim="ademamix", lr=lr, beta1=0.9, beta2=0.999, beta3=b3,
                            alpha=alpha, eps=1e-8, step=k)
        oracle.step(hp, t, g, "f32", 256)
        p_ref = p_ref - lr * (1 + alpha * (1 - b3 ** k)) * gd / (np.abs(gd) + 1e-8)
        np.testing.assert_allclose(t.s1[n:], (1 - b3 ** k) * gd, rtol=2e-5, atol=1e-12)
    np.testing.assert_allclose(t.p, p_ref, rtol=1e-5, atol=2e-7)


def test_ademamix_schedules_endpoints_and_monotone():
    T = 100
    alphas, beta3s = [], []
    for t in range(1, 2 * T):
        sc = oracle.scalars(oracle.HParams(optim="ademamix", alpha=5.0, beta1=0.9, beta3=0.9999,
                                           t_alpha=T, t_beta3=T, step=t))
        alphas.append(sc["alpha_t"])
        beta3s.append(sc["b3t"])
        assert abs(sc["omb3t"] - (1 - sc["b3t"])) <= 1e-7
    alphas, beta3s = np.array(alphas), np.array(beta3s)
    assert np.all(np.diff(alphas) >= 0) and np.all(np.diff(beta3s) >= 0)
    assert alphas[T - 1] == np.float32(5.0) and np.all(alphas[T - 1:] == np.float32(5.0))
    assert alphas[T // 2 - 1] == np.float32(2.5)        # linear warm-up
    assert abs(beta3s[T - 1] - np.float32(0.9999)) <= 1e-7
    assert np.all(beta3s[T:] == np.float32(0.9999))
    # the beta3 warm-up moves the decay half-life linearly: 1/ln(beta3_t) runs from
    # 1/ln(beta1) at t = 0 to 1/ln(beta3) at t = T
    inv_log = 1.0 / np.log(beta3s[:T].astype(np.float64))
    r = np.arange(1, T + 1) / T
    expect = (1 - r) / np.log(np.float64(np.float32(0.9))) + r / np.log(np.float64(np.float32(0.9999)))
    np.testing.assert_allclose(inv_log, expect, rtol=2e-3)
    sc = oracle.scalars(oracle.HParams(optim="ademamix", alpha=5.0, beta3=0.9999, step=7))
    assert sc["alpha_t"] == np.float32(5.0) and sc["b3t"] == np.float32(0.9999)


def test_momentum_constant_gradient_closed_form():
    n, lr, mu = 100, 0.01, 0.9
    g = workloads.normal(n, 1e-2, 50)
    p0 = workloads.normal(n, 0.1, 51)
    t = oracle.TensorState(p0.copy(), np.zeros(n, np.float32), None, None, None, 32)
    p_ref = p0.astype(np.float64)
    for k in range(1, 21):
        oracle.step(oracle.HParams(optim="momentum", lr=lr, beta1=mu, step=k), t, g, "f32", 256)
        m_ref = g.astype(np.float64) * (1 - mu ** k) / (1 - mu)
        p_ref = p_ref - lr * m_ref
        np.testing.assert_allclose(t.s1, m_ref, rtol=1e-5)
    np.testing.assert_allclose(t.p, p_ref, rtol=1e-5, atol=1e-7)


# ---------------------------------------------------------------------------
# the 8-bit step tracks the 32-bit optimizer (benchmark-script method:
# compare, then re-sync p and the 32-bit states to the 8-bit ones)
# ---------------------------------------------------------------------------

TRACK = {
    # optim: (torch comparator or None for the oracle's own 32-bit path, hparams, statenames,
    #         qmaps)
    "adam": (lambda p: torch.optim.Adam([p]), dict(), ["exp_avg", "exp_avg_sq"], (S, U)),
    "adamw": (lambda p: torch.optim.AdamW([p], weight_decay=1e-2), dict(weight_decay=1e-2),
              ["exp_avg", "exp_avg_sq"], (S, U)),
    "momentum": (lambda p: torch.optim.SGD([p], 0.01, 0.9), dict(lr=0.01, beta1=0.9),
                 ["momentum_buffer"], (S, None)),
    "rmsprop": (lambda p: torch.optim.RMSprop([p], 0.01, 0.9), dict(lr=0.01, beta1=0.9),
                ["square_avg"], (U, None)),
    "adagrad": (lambda p: torch.optim.Adagrad([p], 0.01, eps=1e-8), dict(lr=0.01),
                ["sum"], (U, None)),
    "lion": (None, dict(lr=1e-4, beta1=0.9, beta2=0.99), None, (S, None)),
    "ademamix": (None, dict(alpha=5.0, beta3=0.9999, t_alpha=100, t_beta3=100), None, (S, U)),
}


@pytest.mark.parametrize("gtype", ["f32", "bf16"])
@pytest.mark.parametrize("optim", sorted(TRACK))
def test_8bit_step_tracks_32bit(optim, gtype):
    tol = golden("tracking_tolerances.json")
    make, hpkw, names, (q1, q2) = TRACK[optim]
    dim1, dim2 = 64, 256
    n = dim1 * dim2
    B = tol["blocksize"]
    p_init = workloads.normal(n, tol["param_scale"], 60)
    p2 = oracle.to_storage(p_init, gtype)            # 8-bit run holds p in gtype
    p1 = oracle.to_f32(p2, gtype)                    # 32-bit run holds float32
    s1, s2, a1, a2 = oracle.zero_state(optim, n, 8, B, q1, q2)
    t8 = oracle.TensorState(p2, s1, s2, a1, a2, 8)
    if make is not None:
        pt = torch.nn.Parameter(torch.from_numpy(p1.copy()))
        opt = make(pt)
    else:
        r1, r2, _, _ = oracle.zero_state(optim, n, 32, B)
        t32 = oracle.TensorState(p1.copy(), r1, r2, None, None, 32)
    ptol = tol["param"][gtype]
    for k in range(1, 13):
        g = oracle.to_storage(workloads.normal(n, tol["gradient_scale"], 600 + k), gtype)
        g32 = oracle.to_f32(g, gtype)
        hp = oracle.HParams(optim=optim, step=k, **hpkw)
        if make is not None:
            pt.grad = torch.from_numpy(g32.copy())
            opt.step()
            ref_p = pt.detach().numpy().copy()
            ref_states = [opt.state[pt][nm].numpy() for nm in names]
        else:
            oracle.step(hp, t32, g32, "f32", B)
            ref_p = t32.p.copy()
            k_states = oracle.NSTATES[optim]
            ref_states = ([t32.s1[:n], t32.s1[n:], t32.s2] if optim == "ademamix"
                          else [t32.s1] + ([t32.s2] if k_states > 1 else []))
        oracle.step(hp, t8, g, gtype, B, q1, q2)
        p8 = oracle.to_f32(t8.p, gtype)
        # parameters: rtol=patol, atol=prtol as bound by the script's call
        assert np.count_nonzero(~np.isclose(ref_p, p8, rtol=ptol["patol"],
                                            atol=ptol["prtol"])) == 0
        err = np.abs(ref_p - p8)
        relerr = err / (np.abs(ref_p) + 1e-9)
        if gtype == "bf16":
            assert err.mean() <= ptol["err_mean_le"] and relerr.mean() <= ptol["relerr_mean_le"]
        else:
            assert err.mean() < ptol["err_mean_lt"] and relerr.mean() < ptol["relerr_mean_lt"]
        # dequantized states vs the 32-bit states
        deq = []
        if optim == "ademamix":
            nb = n // B
            deq = [oracle.dequantize_blockwise(t8.s1[:n], t8.absmax1[:nb], q1, B),
                   oracle.dequantize_blockwise(t8.s1[n:], t8.absmax1[nb:], q1, B),
                   oracle.dequantize_blockwise(t8.s2, t8.absmax2, q2, B)]
        else:
            deq.append(oracle.dequantize_blockwise(t8.s1, t8.absmax1, q1, B))
            if t8.s2 is not None:
                deq.append(oracle.dequantize_blockwise(t8.s2, t8.absmax2, q2, B))
        for ref, d in zip(ref_states, deq):
            bad = ~np.isclose(ref, d, atol=tol["state"]["atol"], rtol=tol["state"]["rtol"])
            assert np.count_nonzero(bad) < tol["state"]["max_not_close"]
        # re-sync, so that the comparison stays per step
        resync = oracle.to_f32(oracle.to_storage(ref_p, gtype), gtype)
        t8.p[:] = oracle.to_storage(resync, gtype)
        if make is not None:
            with torch.no_grad():
                pt.copy_(torch.from_numpy(resync))
            for nm, d in zip(names, deq):
                opt.state[pt][nm].copy_(torch.from_numpy(d))
        else:
            t32.p[:] = resync
            if optim == "ademamix":
                t32.s1[:n], t32.s1[n:], t32.s2[:] = deq
            else:
                t32.s1[:] = deq[0]


# ---------------------------------------------------------------------------
# skip_zeros (page: 'Support skip_zeros in the XPU Triton optimizer kernels')
# ---------------------------------------------------------------------------

def _random_8bit_state(optim, n, B, seed, q1, q2):
    nb = (n + B - 1) // B
    k = oracle.NSTATES[optim]
    s1 = workloads.random_codes(n * (2 if optim == "ademamix" else 1), seed)
    a1 = workloads.random_absmax(nb * (2 if optim == "ademamix" else 1), 1e-3, seed + 1)
    s2 = a2 = None
    if k >= 2:
        s2 = workloads.random_codes(n, seed + 2)
        a2 = workloads.random_absmax(nb, 1e-6, seed + 3)
    return s1, s2, a1, a2


MAPS = {"adam": (S, U), "adamw": (S, U), "momentum": (S, None), "rmsprop": (U, None),
        "adagrad": (U, None), "lion": (S, None), "ademamix": (S, U)}


@pytest.mark.parametrize("optim", sorted(MAPS))
@pytest.mark.parametrize("state_bits", [8, 32])
@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_skip_zeros_identities(optim, state_bits, dtype):
    q1, q2 = MAPS[optim]
    rows, cols, B = 40, 256, 256
    n = rows * cols
    g = oracle.to_storage(workloads.sparse_rows(rows, cols, 0.25, 1e-2, 70), dtype)
    g32 = oracle.to_f32(g, dtype)
    g32_2 = g32.reshape(rows, cols)
    g32_2[:, 3] = 0.0                                   # zeros inside live rows too
    g = oracle.to_storage(g32, dtype)
    p = oracle.to_storage(workloads.normal(n, 0.1, 71), dtype)
    if state_bits == 8:
        s1, s2, a1, a2 = _random_8bit_state(optim, n, B, 72, q1, q2)
    else:
        s1 = workloads.normal(n * (2 if optim == "ademamix" else 1), 1e-3, 72)
        s2 = np.abs(workloads.normal(n, 1e-3, 73)) if oracle.NSTATES[optim] > 1 else None
        if optim in ("rmsprop", "adagrad"):
            s1 = np.abs(s1)
        a1 = a2 = None
    base = oracle.TensorState(p, s1, s2, a1, a2, state_bits)
    hpkw = dict(optim=optim, step=3, weight_decay=1e-2, alpha=5.0)
    on, off = base.copy(), base.copy()
    oracle.step(oracle.HParams(skip_zeros=True, **hpkw), on, g, dtype, B, q1, q2)
    oracle.step(oracle.HParams(skip_zeros=False, **hpkw), off, g, dtype, B, q1, q2)
    zero = g32 == 0.0
    assert zero.any() and (~zero).any()
    # zero-gradient elements: parameter bit-identical to its pre-step value
    np.testing.assert_array_equal(on.p[zero], base.p[zero])
    # every other element: bit-identical to the skip_zeros=False result
    np.testing.assert_array_equal(on.p[~zero], off.p[~zero])
    if state_bits == 32:
        st_on = [on.s1] + ([on.s2] if on.s2 is not None else [])
        st_base = [base.s1] + ([base.s2] if base.s2 is not None else [])
        st_off = [off.s1] + ([off.s2] if off.s2 is not None else [])
        for so, sb, sf in zip(st_on, st_base, st_off):
            z = np.tile(zero, so.size // n)
            np.testing.assert_array_equal(so[z], sb[z])
            np.testing.assert_array_equal(so[~z], sf[~z])
    else:
        # fully skipped blocks keep codes and absmax; blocks without zeros match skip=False
        blk_all_zero = zero.reshape(-1, B).all(axis=1)
        blk_no_zero = ~zero.reshape(-1, B).any(axis=1)
        assert blk_all_zero.any()
        reps = 2 if optim == "ademamix" else 1
        pairs = [(on.s1, base.s1, off.s1, on.absmax1, base.absmax1, off.absmax1, reps)]
        if on.s2 is not None:
            pairs.append((on.s2, base.s2, off.s2, on.absmax2, base.absmax2, off.absmax2, 1))
        for c_on, c_b, c_off, a_on, a_b, a_off, r in pairs:
            allz, noz = np.tile(blk_all_zero, r), np.tile(blk_no_zero, r)
            np.testing.assert_array_equal(a_on[allz], a_b[allz])
            np.testing.assert_array_equal(c_on.reshape(-1, B)[allz], c_b.reshape(-1, B)[allz])
            np.testing.assert_array_equal(a_on[noz], a_off[noz])
            np.testing.assert_array_equal(c_on.reshape(-1, B)[noz], c_off.reshape(-1, B)[noz])


@pytest.mark.parametrize("optim", sorted(MAPS))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zero_rows_over_zero_states_are_fixed_points(optim, dtype):
    """Without decay, a block whose gradient is all zero (+0 and -0) over zero
    states comes out of a plain step (skip_zeros off) exactly as skip_zeros
    would leave it: p, codes and absmax unchanged.  Every ratio there is a
    signed zero over eps, so the update direction is zero."""
    q1, q2 = MAPS[optim]
    n, B = 8 * 256, 256
    g = workloads.normal(n, 1e-2, 90)
    rng = np.random.default_rng(91)
    zero_blocks = [1, 2, 5]
    for b in zero_blocks:
        g[b * B:(b + 1) * B] = np.where(rng.random(B) < 0.5, 0.0, -0.0)
    g = oracle.to_storage(g, dtype)
    base = oracle.TensorState(oracle.to_storage(workloads.normal(n, 0.1, 92), dtype),
                              *oracle.zero_state(optim, n, 8, B, q1, q2), 8)
    hpkw = dict(optim=optim, step=1, weight_decay=0.0, alpha=5.0)
    on, off = base.copy(), base.copy()
    oracle.step(oracle.HParams(skip_zeros=True, **hpkw), on, g, dtype, B, q1, q2)
    oracle.step(oracle.HParams(skip_zeros=False, **hpkw), off, g, dtype, B, q1, q2)
    for b in zero_blocks:
        sl = slice(b * B, (b + 1) * B)
        np.testing.assert_array_equal(off.p[sl], base.p[sl])
        np.testing.assert_array_equal(off.p[sl], on.p[sl])
    reps = 2 if optim == "ademamix" else 1
    for c_off, c_b, a_off, a_b, r in [(off.s1, base.s1, off.absmax1, base.absmax1, reps),
                                      (off.s2, base.s2, off.absmax2, base.absmax2, 1)]:
        if c_off is None:
            continue
        for k in range(r):
            for b in zero_blocks:
                sl = slice(k * n + b * B, k * n + (b + 1) * B)
                np.testing.assert_array_equal(c_off[sl], c_b[sl])
                assert a_off[k * (n // B) + b] == 0.0
    # the live blocks did move
    assert not np.array_equal(off.p[:B], base.p[:B])


@pytest.mark.parametrize("optim", sorted(MAPS))
def test_skip_zeros_without_zeros_equals_plain(optim):
    q1, q2 = MAPS[optim]
    n, B = 1000, 256
    g = workloads.normal(n, 1e-2, 80)
    g[g == 0] = 1e-3
    s1, s2, a1, a2 = _random_8bit_state(optim, n, B, 81, q1, q2)
    base = oracle.TensorState(workloads.normal(n, 0.1, 82), s1, s2, a1, a2, 8)
    a, b = base.copy(), base.copy()
    oracle.step(oracle.HParams(optim=optim, step=2, skip_zeros=True), a, g, "f32", B, q1, q2)
    oracle.step(oracle.HParams(optim=optim, step=2, skip_zeros=False), b, g, "f32", B, q1, q2)
    for x, y in zip((a.p, a.s1, a.s2, a.absmax1, a.absmax2), (b.p, b.s1, b.s2, b.absmax1,
                                                              b.absmax2)):
        if x is not None:
            np.testing.assert_array_equal(x, y)


# ---------------------------------------------------------------------------
# max_unorm (docs page: "the maximum value to normalize each block with")
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("optim", sorted(MAPS))
def test_max_unorm_invariants(optim):
    q1, q2 = MAPS[optim]
    n, B = 2000, 256
    g = workloads.normal(n, 1e-2, 90)
    s1, s2, a1, a2 = _random_8bit_state(optim, n, B, 91, q1, q2)
    base = oracle.TensorState(workloads.normal(n, 0.02, 92), s1, s2, a1, a2, 8)
    hpkw = dict(optim=optim, step=4, lr=1e-3, alpha=2.0)
    plain, zero_mu, huge_mu, clip = base.copy(), base.copy(), base.copy(), base.copy()
    oracle.step(oracle.HParams(**hpkw), plain, g, "f32", B, q1, q2)
    oracle.step(oracle.HParams(max_unorm=0.0, **hpkw), zero_mu, g, "f32", B, q1, q2)
    r_huge = oracle.step(oracle.HParams(max_unorm=1e30, **hpkw), huge_mu, g, "f32", B, q1, q2)
    assert r_huge == 1.0
    for t in (zero_mu, huge_mu):
        np.testing.assert_array_equal(t.p, plain.p)
        np.testing.assert_array_equal(t.s1, plain.s1)
    # clipping: the applied update norm equals max_unorm * ||p|| (no decay here); the
    # limit is chosen so that the clip halves the step
    _, unorm, pnorm = oracle.unorm_scale(oracle.HParams(max_unorm=1e30, **hpkw), base, g,
                                         "f32", B, q1, q2)
    mu = 0.5 * unorm / pnorm
    scale, _, _ = oracle.unorm_scale(oracle.HParams(max_unorm=mu, **hpkw), base, g, "f32", B,
                                     q1, q2)
    assert abs(scale - 0.5) < 1e-6
    r = oracle.step(oracle.HParams(max_unorm=mu, **hpkw), clip, g, "f32", B, q1, q2)
    assert r == np.float32(scale)
    sc = oracle.scalars(oracle.HParams(**hpkw))
    dp = clip.p.astype(np.float64) - base.p.astype(np.float64)
    applied = np.linalg.norm(dp) / (sc["step_size"]) * sc["unorm_c"]
    assert abs(applied - np.float32(mu) * pnorm) <= 1e-3 * (mu * pnorm)
    # clipping never touches the states
    np.testing.assert_array_equal(clip.s1, plain.s1)
    np.testing.assert_array_equal(clip.absmax1, plain.absmax1)
    # and the update direction is unchanged: dp is parallel to the unclipped step
    dp0 = plain.p.astype(np.float64) - base.p.astype(np.float64)
    cos = dp.dot(dp0) / (np.linalg.norm(dp) * np.linalg.norm(dp0))
    assert cos > 1 - 1e-6


def test_max_unorm_norms_match_numpy():
    # the norms the clip uses, against a numpy evaluation for Momentum (u = m)
    n = 3000
    g = workloads.normal(n, 1e-2, 95)
    p = workloads.normal(n, 0.02, 96)
    m0 = workloads.normal(n, 1e-2, 97)
    t = oracle.TensorState(p, m0.copy(), None, None, None, 32)
    hp = oracle.HParams(optim="momentum", lr=0.01, beta1=0.9, max_unorm=0.5, step=2)
    scale, unorm, pnorm = oracle.unorm_scale(hp, t, g, "f32", 256)
    m_new = 0.9 * m0.astype(np.float64) + g
    assert abs(unorm - np.linalg.norm(m_new)) <= 1e-6 * unorm
    assert abs(pnorm - np.linalg.norm(p.astype(np.float64))) <= 1e-12 * pnorm
    expect = 0.5 * pnorm / unorm if unorm > 0.5 * pnorm else 1.0
    assert abs(scale - expect) <= 1e-6 * expect


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_param_sumsq_closed_forms(dtype):
    # Pythagorean quadruples and sign: every value is exact in all three dtypes
    p = oracle.to_storage(np.array([2.0, -3.0, 6.0, 1.0, -2.0, 2.0], np.float32), dtype)
    assert oracle.param_sumsq(p, dtype) == 4 + 9 + 36 + 1 + 4 + 4
    ones = oracle.to_storage(np.full(1000, -0.5, np.float32), dtype)
    assert oracle.param_sumsq(ones, dtype) == 250.0
    assert oracle.param_sumsq(oracle.to_storage(np.zeros(0, np.float32), dtype), dtype) == 0.0
    # the squares are taken of the stored values (rounded to the dtype), not of
    # the binary32 inputs
    x = np.array([1.0 + 2.0 ** -12], np.float32)
    stored = float(oracle.to_f32(oracle.to_storage(x, dtype), dtype)[0])
    assert oracle.param_sumsq(oracle.to_storage(x, dtype), dtype) == stored * stored
    if dtype != "f32":
        assert stored == 1.0


def test_param_sumsq_matches_an_exactly_rounded_sum():
    p = workloads.normal(100000, 0.02, 140)
    exact = math.fsum(float(v) * float(v) for v in p.astype(np.float64))
    got = oracle.param_sumsq(p, "f32")
    # n * 2^-53 relative bound of a recursive binary64 sum of positive terms
    assert abs(got - exact) <= 100000 * 2.0 ** -53 * exact


@pytest.mark.parametrize("optim,wd", [("adam", 0.0), ("adam", 0.1), ("adamw", 0.1),
                                      ("momentum", 0.0), ("lion", 0.1), ("ademamix", 0.1)])
def test_next_step_norm_is_the_norm_this_step_leaves(optim, wd):
    # the norm a step can carry forward: after step k, the P of step k + 1's
    # max_unorm test is the norm of the p step k wrote (decay included)
    q1, q2 = MAPS[optim]
    n, B = 1500, 256
    s1, s2, a1, a2 = _random_8bit_state(optim, n, B, 141, q1, q2)
    t = oracle.TensorState(workloads.normal(n, 0.02, 142), s1, s2, a1, a2, 8)
    hpkw = dict(optim=optim, lr=1e-3, alpha=2.0, weight_decay=wd, max_unorm=0.05)
    for k in (1, 2, 3):
        oracle.step(oracle.HParams(step=k, **hpkw), t, workloads.normal(n, 1e-2, 143 + k),
                    "f32", B, q1, q2)
        _, _, pnorm = oracle.unorm_scale(oracle.HParams(step=k + 1, **hpkw), t,
                                         workloads.normal(n, 1e-2, 150 + k), "f32", B, q1, q2)
        want = np.linalg.norm(t.p.astype(np.float64))
        assert abs(pnorm - want) <= 1e-12 * want
        assert pnorm == math.sqrt(oracle.param_sumsq(t.p, "f32"))


@pytest.mark.parametrize("optim,wd,depends", [("adam", 0.0, False), ("adam", 0.1, True),
                                              ("adamw", 0.1, False), ("lion", 0.1, False),
                                              ("momentum", 0.1, True),
                                              ("ademamix", 0.1, False)])
def test_update_norm_depends_on_p_only_through_coupled_decay(optim, wd, depends):
    # the reading that lets a pre-pass with a carried ||p|| skip reading p: the
    # update direction's norm U involves p only through weight decay added to
    # the gradient (coupled); decoupled decay is applied to p after the
    # direction, outside U
    q1, q2 = MAPS[optim]
    n, B = 1200, 256
    s1, s2, a1, a2 = _random_8bit_state(optim, n, B, 160, q1, q2)
    g = workloads.normal(n, 1e-2, 161)
    hp = oracle.HParams(optim=optim, lr=1e-3, alpha=2.0, weight_decay=wd, max_unorm=0.05,
                        step=3)
    us = []
    for seed in (162, 163):
        t = oracle.TensorState(workloads.normal(n, 0.5, seed), s1.copy(),
                               None if s2 is None else s2.copy(), a1.copy(),
                               None if a2 is None else a2.copy(), 8)
        us.append(oracle.unorm_scale(hp, t, g, "f32", B, q1, q2)[1])
    if depends:
        assert abs(us[0] - us[1]) > 1e-6 * us[0]
    else:
        assert us[0] == us[1]


@pytest.mark.parametrize("optim,bits", [("adam", 8), ("momentum", 8), ("lion", 8),
                                         ("adam", 32)])
def test_max_unorm_per_block_invariants(optim, bits):
    # the per-block reading: every block of B elements gets its own multiplier
    q1, q2 = MAPS[optim]
    n, B = 2000, 256
    nb = (n + B - 1) // B
    g = workloads.normal(n, 1e-2, 130)
    if bits == 8:
        s1, s2, a1, a2 = _random_8bit_state(optim, n, B, 131, q1, q2)
    else:
        s1 = workloads.normal(n, 1e-3, 131)
        s2 = np.abs(workloads.normal(n, 1e-4, 132)) if oracle.NSTATES[optim] == 2 else None
        a1 = a2 = None
    base = oracle.TensorState(workloads.normal(n, 0.02, 133), s1, s2, a1, a2, bits)
    hpkw = dict(optim=optim, step=3, lr=1e-3)

    def block(t, b):
        lo, hi = b * B, min(n, (b + 1) * B)
        sl = lambda x: None if x is None else x[lo:hi]
        am = lambda x: None if x is None else x[b:b + 1]
        return oracle.TensorState(t.p[lo:hi].copy(), sl(t.s1).copy(),
                                  None if t.s2 is None else sl(t.s2).copy(),
                                  None if t.absmax1 is None else am(t.absmax1).copy(),
                                  None if t.absmax2 is None else am(t.absmax2).copy(), bits)

    # per-block norms, each block taken as a tensor of its own
    U, P = np.zeros(nb), np.zeros(nb)
    for b in range(nb):
        _, U[b], P[b] = oracle.unorm_scale(oracle.HParams(max_unorm=1e30, **hpkw), block(base, b),
                                           g[b * B:(b + 1) * B], "f32", B, q1, q2)
    mu = float(np.median(U / P))   # about half of the blocks get clipped
    plain, off, clip = base.copy(), base.copy(), base.copy()
    oracle.step(oracle.HParams(**hpkw), plain, g, "f32", B, q1, q2)
    oracle.step(oracle.HParams(max_unorm=0.0, unorm_per_block=True, **hpkw), off, g, "f32", B,
                q1, q2)
    oracle.step(oracle.HParams(max_unorm=mu, unorm_per_block=True, **hpkw), clip, g, "f32", B,
                q1, q2)
    np.testing.assert_array_equal(off.p, plain.p)
    # clipping never touches the states
    for name in ("s1", "s2", "absmax1", "absmax2"):
        if getattr(plain, name) is not None:
            np.testing.assert_array_equal(getattr(clip, name), getattr(plain, name))
    sc = oracle.scalars(oracle.HParams(**hpkw))
    clipped = 0
    for b in range(nb):
        lo, hi = b * B, min(n, (b + 1) * B)
        dp = clip.p[lo:hi].astype(np.float64) - base.p[lo:hi].astype(np.float64)
        dp0 = plain.p[lo:hi].astype(np.float64) - base.p[lo:hi].astype(np.float64)
        if U[b] > np.float32(mu) * P[b]:
            clipped += 1
            applied = np.linalg.norm(dp) / sc["step_size"] * sc["unorm_c"]
            assert abs(applied - np.float32(mu) * P[b]) <= 1e-3 * (mu * P[b]), b
            assert dp.dot(dp0) / (np.linalg.norm(dp) * np.linalg.norm(dp0)) > 1 - 1e-6
        else:
            np.testing.assert_array_equal(clip.p[lo:hi], plain.p[lo:hi])
    assert 0 < clipped < nb


def test_max_unorm_per_block_equals_per_tensor_on_one_block():
    # a tensor of one block: the two readings take the same norms
    q1, q2 = MAPS["adam"]
    n = B = 256
    g = workloads.normal(n, 1e-2, 140)
    s1, s2, a1, a2 = _random_8bit_state("adam", n, B, 141, q1, q2)
    base = oracle.TensorState(workloads.normal(n, 0.02, 142), s1, s2, a1, a2, 8)
    hpkw = dict(optim="adam", step=5, lr=1e-3, weight_decay=1e-2)
    _, unorm, pnorm = oracle.unorm_scale(oracle.HParams(max_unorm=1e30, **hpkw), base, g, "f32",
                                         B, q1, q2)
    mu = 0.3 * unorm / pnorm
    a, b = base.copy(), base.copy()
    oracle.step(oracle.HParams(max_unorm=mu, **hpkw), a, g, "f32", B, q1, q2)
    oracle.step(oracle.HParams(max_unorm=mu, unorm_per_block=True, **hpkw), b, g, "f32", B, q1, q2)
    for x, y in zip((a.p, a.s1, a.s2, a.absmax1, a.absmax2), (b.p, b.s1, b.s2, b.absmax1, b.absmax2)):
        np.testing.assert_array_equal(x, y)
    assert not np.array_equal(a.p, base.p)


# ---------------------------------------------------------------------------
# checkpoint round trip (benchmark script: save/load the state every 10 steps;
# raw codes and qmap must be identical after reload)
# ---------------------------------------------------------------------------

def test_checkpoint_round_trip_is_bit_identical(tmp_path):
    n, B = 5000, 256
    s1, s2, a1, a2 = oracle.zero_state("adam", n, 8, B, S, U)
    straight = oracle.TensorState(workloads.normal(n, 0.1, 110), s1, s2, a1, a2, 8)
    resumed = straight.copy()
    grads = [workloads.normal(n, 0.01, 120 + k) for k in range(1, 21)]
    for k in range(1, 21):
        hp = oracle.HParams(optim="adam", step=k)
        oracle.step(hp, straight, grads[k - 1], "f32", B, S, U)
        oracle.step(hp, resumed, grads[k - 1], "f32", B, S, U)
        if k % 10 == 0:
            path = tmp_path / f"opt{k}.npz"
            np.savez(path, p=resumed.p, s1=resumed.s1, s2=resumed.s2, a1=resumed.absmax1,
                     a2=resumed.absmax2, q1=S, q2=U)
            del resumed
            z = np.load(path)
            resumed = oracle.TensorState(z["p"].copy(), z["s1"].copy(), z["s2"].copy(),
                                         z["a1"].copy(), z["a2"].copy(), 8)
            np.testing.assert_array_equal(z["q1"], S)
            np.testing.assert_array_equal(resumed.s1, straight.s1)
    for x, y in zip((straight.p, straight.s1, straight.s2, straight.absmax1, straight.absmax2),
                    (resumed.p, resumed.s1, resumed.s2, resumed.absmax1, resumed.absmax2)):
        np.testing.assert_array_equal(x, y)
