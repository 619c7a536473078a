"""Failure detection of the step kernel's bounded waits, without a GPU fault.

The plain step streams each warp's chunks through shared memory with
asynchronous bulk copies and waits for them on mbarriers.  Every such wait
is bounded (1 s): instead of hanging, a warp whose copy never lands records
BNB8_STATUS_WAIT_TIMEOUT in the library's device status word, stops
computing and returns.  The test hook BNB8_TEST_STALL_WAIT makes one warp
withhold its own first copy, so that its wait runs out; the call must then
come back with the status set, and the device must stay usable: the next
step, on fresh state, matches the oracle bit for bit."""
import numpy as np
import pytest

import oracle
import workloads
from parity_util import assert_same, maps, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

S, U = maps()


@pytest.fixture(scope="module")
def bnb8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_block_wise_gb300 as m
    from bit_block_wise_gb300 import build
    build.build()
    m.lib()
    return m


def _params(bnb8, n, seed):
    p = workloads.normal(n, 0.02, seed)
    st = oracle.zero_state("adam", n, 8, 256, S, U)
    ps = bnb8.ParamState(to_dev(p), to_dev(workloads.normal(n, 1e-3, seed + 1)),
                         *[to_dev(x) for x in st], 8)
    return ps, oracle.TensorState(p.copy(), *st, 8)


def test_stalled_copy_sets_the_status_and_the_device_recovers(bnb8):
    qd1, qd2 = to_dev(S), to_dev(U)
    assert bnb8.bnb8_device_status(clear=True) in (0, bnb8.BNB8_STATUS_WAIT_TIMEOUT)
    assert bnb8.bnb8_device_status() == 0
    n = 256 * 4096
    ps, _ = _params(bnb8, n, 3)
    hp = bnb8.HParams(optim="adam", step=1, extra_flags=bnb8.BNB8_TEST_STALL_WAIT)
    bnb8.bnb8_step_2state([ps], hp, qd1, qd2)
    torch.cuda.synchronize()
    assert bnb8.bnb8_device_status(clear=True) == bnb8.BNB8_STATUS_WAIT_TIMEOUT
    assert bnb8.bnb8_device_status() == 0
    # the context is intact: a plain step on fresh state equals the oracle
    ps, ref = _params(bnb8, n, 5)
    g = to_host(ps.g)
    bnb8.bnb8_step_2state([ps], bnb8.HParams(optim="adam", step=1), qd1, qd2)
    torch.cuda.synchronize()
    oracle.step(oracle.HParams(optim="adam", step=1), ref, g, "f32", 256, S, U)
    assert bnb8.bnb8_device_status() == 0
    assert_same("p", to_host(ps.p), ref.p)
    assert_same("s1", to_host(ps.s1), ref.s1)
    assert_same("s2", to_host(ps.s2), ref.s2)
    assert_same("absmax1", to_host(ps.absmax1), ref.absmax1)
    assert_same("absmax2", to_host(ps.absmax2), ref.absmax2)


def test_unknown_flag_bits_are_rejected(bnb8):
    p = torch.zeros(1024, device="cuda")
    ps = bnb8.ParamState(p, torch.zeros_like(p), *bnb8.zero_state(p, "adam"), 8)
    with pytest.raises(bnb8.Bnb8Error):
        bnb8.bnb8_step_2state([ps], bnb8.HParams(optim="adam", extra_flags=0x200), to_dev(S), to_dev(U))
