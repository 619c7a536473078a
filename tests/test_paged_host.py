"""Paged-state host logic without a GPU: the shared-buffer layout of
paged_zero_states, the optimizer packing the states it creates into one
buffer, and paged_prefetch moving each buffer once.  The managed allocation
is replaced by host memory and the C prefetch call by a recorder."""
import pytest
import torch

import bit_block_wise_gb300 as bnb8
from bit_block_wise_gb300 import optim as O


@pytest.fixture
def host_paged(monkeypatch):
    monkeypatch.setattr(bnb8, "paged_empty",
                        lambda count, dtype, device=None: torch.empty(count, dtype=dtype))


SPECS = [(5000, "adam", 8, 256), (100, "adam", 32, 256), (3 * 256 + 7, "ademamix", 8, 256),
         (4096, "rmsprop", 8, 0), (777, "lion", 8, 64)]


def test_paged_zero_states_layout(host_paged):
    ps = [torch.zeros(n) for n, *_ in SPECS]
    got = bnb8.paged_zero_states([(p, o, b, B) for p, (n, o, b, B) in zip(ps, SPECS)])
    base = None
    ends = []
    for p, (n, o, b, B), arrays in zip(ps, SPECS, got):
        want = bnb8.zero_state(p, o, b, B)
        for t, w in zip(arrays, want):
            assert (t is None) == (w is None)
            if t is None:
                continue
            assert t.dtype == w.dtype and torch.equal(t, w)
            st = t.untyped_storage()
            base = st.data_ptr() if base is None else base
            assert st.data_ptr() == base                     # one buffer for all
            off = t.data_ptr() - base
            assert off % 256 == 0                             # aligned slices
            ends.append((off, off + t.numel() * t.element_size()))
    ends.sort()
    assert all(a[1] <= b[0] for a, b in zip(ends, ends[1:]))  # no overlap


def test_optimizer_packs_new_states_into_one_buffer(host_paged):
    params = [torch.nn.Parameter(torch.zeros(n)) for n in (8192, 100, 5000)]
    opt = O.PagedAdamW8bit(params, manager=O.OptimManager())
    g = opt.param_groups[0]
    opt._init_states([(p, opt._config(g, p)) for p in params])
    bufs = {t.untyped_storage().data_ptr() for p in params for t in opt.state[p].values()
            if torch.is_tensor(t)}
    assert len(bufs) == 1
    assert [opt.state[p]["state_bits"] for p in params] == [8, 32, 8]
    assert torch.all(opt.state[params[0]]["state1"] == 127)
    assert torch.all(opt.state[params[0]]["state2"] == 0)


def test_paged_prefetch_moves_each_buffer_once(host_paged, monkeypatch):
    calls = []

    class FakeLib:
        def bnb8_paged_prefetch(self, ptr, nbytes, dev, stream):
            calls.append((ptr, nbytes, dev, stream))
            return bnb8.BNB8_OK

    monkeypatch.setattr(bnb8, "lib", lambda: FakeLib())
    a = bnb8.paged_zero_states([(torch.zeros(5000), "adam", 8, 256)])[0]
    b = bnb8.paged_zero_states([(torch.zeros(300), "lion", 8, 256)])[0]
    bnb8.paged_prefetch(list(a) + list(b) + [None], device=0, stream=7)
    assert len(calls) == 2
    for arrays, call in zip((a, b), calls):
        st = arrays[0].untyped_storage()
        assert call == (st.data_ptr(), st.nbytes(), 0, 7)
    calls.clear()
    bnb8.paged_prefetch(a[0], device="cpu", stream=7)
    assert calls == [(a[0].untyped_storage().data_ptr(), a[0].untyped_storage().nbytes(),
                      bnb8.BNB8_PAGED_HOST, 7)]
