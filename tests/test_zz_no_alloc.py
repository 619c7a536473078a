"""bnb8_unorm_static: the max_unorm pre-pass for callers that cannot allocate
device memory (every byte handed out by a host framework's pool, or a hot loop
where cudaMalloc / cudaFree would stall the device).  It keeps its partial
norms in a fixed scratch array inside the library instead of a caller
workspace.  It must give bnb8_unorm's (workspace) results bit for bit, and the
oracle's multipliers to 1e-6, call after call, although the array keeps
whatever the previous call left in it.

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest

import oracle
import workloads
from parity_util import map_pair, maps, random_state, to_dev, to_host

S, U = maps()
FAKE = 0x7f0000000000  # never dereferenced: the case below fails validation first


@pytest.fixture(scope="module")
def bnb8():
    import bit_block_wise_gb300 as m
    from bit_block_wise_gb300 import build
    build.build()
    m.lib()
    return m


def _tensor_list(bnb8, optim, sizes, bits, seed, p_scale=1.0):
    q1, q2 = map_pair(optim, S, U)
    params, refs = [], []
    for i, (n, b) in enumerate(zip(sizes, bits)):
        st = random_state(optim, n, b, 256, seed + 10 * i, q1, q2)
        p = (workloads.normal(n, 0.02, seed + 10 * i + 5) * np.float32(p_scale)).astype(np.float32)
        g = workloads.normal(n, 1e-2, seed + 10 * i + 6)
        refs.append((oracle.TensorState(p.copy(), *st, b), g))
        params.append(bnb8.ParamState(to_dev(p), to_dev(g), *[to_dev(a) for a in st], b))
    return params, refs, q1, q2


def _out(n):
    import torch
    return torch.empty(n, dtype=torch.float32, device="cuda")


@pytest.mark.gpu
@pytest.mark.parametrize("optim", ["adam", "momentum", "ademamix"])
def test_static_scratch_matches_workspace_version_and_oracle_twice(bnb8, optim):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hp = dict(optim=optim, max_unorm=0.02, step=4, lr=1e-3, beta1=0.9, beta2=0.999, alpha=2.0)
    bhp, ohp = bnb8.HParams(**hp), oracle.HParams(**hp)
    # First call: parameters of 1e30 make every partial norm of this call
    # non-finite (p^2 overflows), so that the second, smaller list would
    # change its multipliers if it read any partial it did not write itself.
    params, _, q1, q2 = _tensor_list(bnb8, optim, [70000, 700, 256 * 300 + 3], [8, 32, 8], 100,
                                     p_scale=5e31)
    qd1 = to_dev(q1)
    qd2 = None if q2 is None else to_dev(q2)
    first_ws = bnb8.bnb8_unorm(params, bhp, qd1, qd2)
    first = bnb8.bnb8_unorm_static(params, bhp, qd1, qd2, out_scale=_out(len(params)))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_host(first), to_host(first_ws))
    # Second call: an ordinary list with fewer blocks than the first wrote.
    params, refs, q1, q2 = _tensor_list(bnb8, optim, [5000, 1234], [8, 8], 200)
    want = bnb8.bnb8_unorm(params, bhp, qd1, qd2)
    got = bnb8.bnb8_unorm_static(params, bhp, qd1, qd2, out_scale=_out(len(params)))
    torch.cuda.synchronize()
    w, gt = to_host(want), to_host(got)
    np.testing.assert_array_equal(gt, w)             # same kernels and summation order
    assert np.all(w < 1.0)                           # the clip is active in this case
    for i, (ref, g) in enumerate(refs):
        scale, _, _ = oracle.unorm_scale(ohp, ref, g, "f32", 256, q1, q2)
        assert abs(float(gt[i]) - scale) <= 1e-6 * scale, (i, float(gt[i]), scale)


def test_static_scratch_needs_an_output_buffer(bnb8):
    with pytest.raises(ValueError):
        bnb8.bnb8_unorm_static([], bnb8.HParams(max_unorm=1.0), None)


def test_static_scratch_rejects_lists_beyond_its_size(bnb8):
    L = bnb8.lib()
    n = (262144 + 1) * 256                           # one block more than the array holds
    t = bnb8.Bnb8Tensor(FAKE, FAKE + 4096, FAKE + 8192, FAKE + 12288, FAKE + 16384,
                        FAKE + 20480, n, 8, 0)
    arr = (bnb8.Bnb8Tensor * 1)(t)
    hp = bnb8.HParams(optim="adam", max_unorm=1.0).c(bnb8.BNB8_F32)
    rc = L.bnb8_unorm_static(arr, 1, ctypes.byref(hp), FAKE, FAKE, FAKE, None)
    assert rc == bnb8.BNB8_EWORKSPACE
    assert b"262144" in L.bnb8_last_error()
