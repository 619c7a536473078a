"""Non-finite values through the step, against the oracle.

The pages fix no rule for NaN or infinity; the oracle's readings are that a
block's absmax is the IEEE 754-2019 maximum (NaN when any new state of the
block is NaN, infinite when one is infinite), that the reciprocal of a NaN
or infinite absmax is 0, and that everything else is IEEE binary32
arithmetic.  Gradients holding NaN, +inf and -inf, parameters holding +0 and
-0, and (for Lion, whose step term the kernels form by bits) zero first
moments and an infinite learning rate go through every kernel family: the
dense ring (B = 256 and 2048), the skip_zeros ring, the register-streaming
kernel (B = 128) and binary32 states.  Values must match bit for bit, except
that any NaN matches any NaN (payloads differ between the host's C library
and the GPU)."""
import numpy as np
import pytest

import oracle
import workloads
from parity_util import map_pair, maps, random_state, to_dev, to_host

S, U = maps()
pytestmark = pytest.mark.gpu

HP = {
    "adam": dict(lr=1e-3, beta1=0.9, beta2=0.999),
    "momentum": dict(lr=0.01, beta1=0.9),
    "rmsprop": dict(lr=0.01, beta1=0.9),
    "lion": dict(lr=1e-4, beta1=0.9, beta2=0.99),
    "ademamix": dict(lr=1e-3, beta1=0.9, beta2=0.999, beta3=0.9999, alpha=5.0, t_alpha=10,
                     t_beta3=10),
}


@pytest.fixture(scope="module")
def bnb8():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_block_wise_gb300 as m
    from bit_block_wise_gb300 import build
    build.build()
    m.lib()
    return m


def _same(name, got, want, dtype=None):
    """Bit-equal, any NaN equal to any NaN."""
    if got is None and want is None:
        return
    assert got.shape == want.shape, name
    if dtype in ("bf16", "f16"):
        gv, wv = oracle.to_f32(got, dtype), oracle.to_f32(want, dtype)
        gb, wb = got, want
    elif got.dtype == np.float32:
        gv, wv = got, want
        gb, wb = got.view(np.uint32), want.view(np.uint32)
    else:
        gv = wv = None
        gb, wb = got, want
    if gv is not None:
        gn, wn = np.isnan(gv), np.isnan(wv)
        bad = np.flatnonzero((gn != wn) | (~gn & (gb != wb)))
    else:
        bad = np.flatnonzero(gb != wb)
    if bad.size:
        i = bad[0]
        raise AssertionError(f"{name}: {bad.size} of {got.size} differ; first at {i}: "
                             f"got {got[i]!r} want {want[i]!r}")


def _grad(n, k, dtype, seed):
    g = workloads.normal(n, 1e-2, seed + 100 * k)
    rng = np.random.default_rng(seed + k)
    idx = rng.choice(n, size=9, replace=False)
    g[idx[:3]] = np.nan
    g[idx[3:5]] = np.inf
    g[idx[5:7]] = -np.inf
    g[idx[7]] = 0.0
    g[idx[8]] = -0.0
    return oracle.to_storage(g, dtype)


def _run(bnb8, optim, dtype, bits, B, n, steps=2, skip_zeros=False, init="random", lr=None,
         seed=70):
    q1, q2 = map_pair(optim, S, U)
    qd1 = to_dev(q1)
    qd2 = None if q2 is None else to_dev(q2)
    p = workloads.normal(n, 0.1, seed)
    p[::37] = 0.0
    p[5::41] = -0.0
    p = oracle.to_storage(p, dtype)
    if init == "zero":
        st = oracle.zero_state(optim, n, bits, B, q1, q2)
    else:
        st = random_state(optim, n, bits, B, seed + 1, q1, q2)
    ref = oracle.TensorState(p.copy(), *[None if a is None else a.copy() for a in st], bits)
    ps = bnb8.ParamState(to_dev(p, dtype), None, *[to_dev(a) for a in st], bits)
    for k in range(1, steps + 1):
        hp = dict(HP[optim], step=k, skip_zeros=skip_zeros)
        if lr is not None:
            hp["lr"] = lr
        g = _grad(n, k, dtype, seed)
        ps.g = to_dev(g, dtype)
        bnb8.step([ps], bnb8.HParams(optim=optim, blocksize=B, **hp), qd1, qd2)
        oracle.step(oracle.HParams(optim=optim, **hp), ref, g, dtype, B, q1, q2)
        import torch
        torch.cuda.synchronize()
        tag = f"{optim}/{dtype}/bits{bits}/B{B}/skip{int(skip_zeros)}/{init}/step{k}"
        _same(tag + " p", to_host(ps.p), ref.p, dtype)
        _same(tag + " s1", to_host(ps.s1), ref.s1)
        _same(tag + " s2", to_host(ps.s2), ref.s2)
        _same(tag + " absmax1", to_host(ps.absmax1), ref.absmax1)
        _same(tag + " absmax2", to_host(ps.absmax2), ref.absmax2)


@pytest.mark.parametrize("optim", ["adam", "momentum", "rmsprop", "lion", "ademamix"])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("B", [256, 2048])
def test_nonfinite_gradients_on_the_ring(bnb8, optim, dtype, B):
    _run(bnb8, optim, dtype, 8, B, 5 * B + 77)


@pytest.mark.parametrize("optim", ["adam", "momentum", "lion"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_nonfinite_gradients_with_skip_zeros(bnb8, optim, dtype):
    _run(bnb8, optim, dtype, 8, 256, 6 * 512 + 100, skip_zeros=True)


@pytest.mark.parametrize("optim", ["adam", "lion"])
@pytest.mark.parametrize("bits,B", [(8, 128), (32, 256)])
def test_nonfinite_gradients_other_kernels(bnb8, optim, bits, B):
    _run(bnb8, optim, "f32", bits, B, 3000)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("skip_zeros", [False, True])
def test_lion_zero_moments_over_signed_zero_parameters(bnb8, dtype, skip_zeros):
    """From zero states a zero gradient gives c = +-0: the step term is the
    signed zero -eff * (+0), which decides the sign of a zero parameter."""
    _run(bnb8, "lion", dtype, 8, 256, 4 * 512 + 33, skip_zeros=skip_zeros, init="zero")


@pytest.mark.parametrize("skip_zeros", [False, True])
def test_lion_infinite_learning_rate(bnb8, skip_zeros):
    """-inf * sign(c): infinite where |c| > 0, NaN where c is zero or NaN."""
    _run(bnb8, "lion", "f32", 8, 256, 3 * 512 + 9, steps=1, skip_zeros=skip_zeros, lr=np.inf)
