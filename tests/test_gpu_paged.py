"""Paged optimizer state on the GPU: state arrays in managed memory
(bnb8_paged_alloc), moved between host and device by bnb8_paged_prefetch,
step bit-identically to device-resident states, through the library and
through the Paged* optimizer classes, including states paged out to the host
between steps and a state_dict round trip."""
import copy

import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bnb8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_block_wise_gb300 as m
    m.lib()
    return m


def test_paged_buffer_round_trip(bnb8):
    t = bnb8.paged_empty(1 << 20, torch.float32)
    assert t.is_cuda and t.dtype == torch.float32 and t.numel() == 1 << 20
    t.copy_(torch.arange(1 << 20, dtype=torch.float32, device="cuda"))
    bnb8.paged_prefetch(t, "cpu")
    torch.cuda.synchronize()
    bnb8.paged_prefetch(t)
    assert torch.equal(t, torch.arange(1 << 20, dtype=torch.float32, device="cuda"))


@pytest.mark.parametrize("optim,dtype,bits", [("adam", torch.float32, 8), ("adamw", torch.bfloat16, 8),
                                              ("lion", torch.bfloat16, 8), ("rmsprop", torch.float16, 8),
                                              ("ademamix", torch.float32, 8), ("adam", torch.float32, 32)])
@pytest.mark.parametrize("evict", [False, True])
def test_paged_states_step_bit_identically(bnb8, optim, dtype, bits, evict):
    n = 3 * 4096 + 40  # several blocks and a ragged tail
    dev = torch.device("cuda")
    p0 = workloads.torch_normal(n, 0.1, 5, dev, dtype)
    q1 = bnb8.bnb8_create_qmap(optim not in ("rmsprop", "adagrad")).to(dev)
    q2 = bnb8.bnb8_create_qmap(False).to(dev)
    runs = []
    for paged in (False, True):
        p = p0.clone()
        s1, s2, a1, a2 = bnb8.zero_state(p, optim, bits, 256, paged=paged)
        ps = bnb8.ParamState(p, None, s1, s2, a1, a2, bits)
        for k in range(1, 4):
            ps.g = workloads.torch_normal(n, 1e-2, 100 + k, dev, dtype)
            if paged:
                if evict:  # paged out to the host since the last step
                    bnb8.paged_prefetch([s1, s2, a1, a2], "cpu")
                bnb8.paged_prefetch([s1, s2, a1, a2])
            bnb8.step([ps], bnb8.HParams(optim=optim, step=k, weight_decay=1e-2,
                                         alpha=5.0 if optim == "ademamix" else 0.0), q1, q2)
        torch.cuda.synchronize()
        runs.append([t.clone() for t in (p, s1, s2, a1, a2) if t is not None])
    for a, b in zip(*runs):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_paged_step_matches_oracle(bnb8):
    """Adam8bit on paged states against the oracle (codes, absmax and p exact)."""
    n, B = 5000, 256
    dev = torch.device("cuda")
    S = oracle.create_qmap(True)
    U = oracle.create_qmap(False)
    p_host = workloads.normal(n, 0.1, 9).astype(np.float32)
    ref = oracle.TensorState(p_host.copy(), *oracle.zero_state("adam", n, 8, B, S, U), 8)
    p = torch.from_numpy(p_host.copy()).to(dev)
    s1, s2, a1, a2 = bnb8.zero_state(p, "adam", 8, B, paged=True)
    ps = bnb8.ParamState(p, None, s1, s2, a1, a2, 8)
    q1, q2 = torch.from_numpy(S).to(dev), torch.from_numpy(U).to(dev)
    for k in range(1, 4):
        g = workloads.normal(n, 1e-2, 50 + k).astype(np.float32)
        ps.g = torch.from_numpy(g).to(dev)
        bnb8.paged_prefetch([s1, s2, a1, a2], "cpu")
        bnb8.paged_prefetch([s1, s2, a1, a2])
        hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, step=k)
        bnb8.step([ps], bnb8.HParams(optim="adam", blocksize=B, **hp), q1, q2)
        oracle.step(oracle.HParams(optim="adam", **hp), ref, g, "f32", B, S, U)
    torch.cuda.synchronize()
    assert np.array_equal(p.cpu().numpy().view(np.uint32), ref.p.view(np.uint32))
    assert np.array_equal(s1.cpu().numpy(), ref.s1)
    assert np.array_equal(s2.cpu().numpy(), ref.s2)
    assert np.array_equal(a1.cpu().numpy().view(np.uint32), ref.absmax1.view(np.uint32))
    assert np.array_equal(a2.cpu().numpy().view(np.uint32), ref.absmax2.view(np.uint32))


def test_paged_zero_states_share_one_buffer(bnb8):
    """Several parameters' states in one paged buffer: aligned slices holding
    the zero codes, stepped as one list bit-identically to device states."""
    dev = torch.device("cuda")
    sizes, bits = [5000, 100, 3 * 256 + 7, 4096], [8, 32, 8, 8]
    ps = [workloads.torch_normal(n, 0.1, 30 + i, dev, torch.bfloat16) for i, n in enumerate(sizes)]
    paged = bnb8.paged_zero_states([(p, "adamw", b, 256) for p, b in zip(ps, bits)])
    storages = {t.untyped_storage().data_ptr() for st in paged for t in st if t is not None}
    assert len(storages) == 1
    for st, p, b in zip(paged, ps, bits):
        for t, want in zip(st, bnb8.zero_state(p, "adamw", b, 256)):
            assert (t is None) == (want is None)
            if t is not None:
                assert t.data_ptr() % 256 == 0 and torch.equal(t, want)
    q1, q2 = bnb8.bnb8_create_qmap(True).to(dev), bnb8.bnb8_create_qmap(False).to(dev)
    runs = []
    for use_paged in (False, True):
        p_run = [p.clone() for p in ps]
        states = paged if use_paged else [bnb8.zero_state(p, "adamw", b, 256) for p, b in zip(ps, bits)]
        plist = [bnb8.ParamState(p, None, *st, b) for p, st, b in zip(p_run, states, bits)]
        for k in range(1, 4):
            for i, ps_ in enumerate(plist):
                ps_.g = workloads.torch_normal(sizes[i], 1e-2, 500 + 10 * k + i, dev, torch.bfloat16)
            if use_paged:
                bnb8.paged_prefetch([t for st in states for t in st], "cpu")
                bnb8.paged_prefetch([t for st in states for t in st])
            bnb8.step(plist, bnb8.HParams(optim="adamw", step=k, weight_decay=1e-2), q1, q2)
        torch.cuda.synchronize()
        runs.append([t.clone() for ps_ in plist for t in (ps_.p, ps_.s1, ps_.s2, ps_.absmax1, ps_.absmax2)
                     if t is not None])
    for a, b in zip(*runs):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def _model(seed):
    torch.manual_seed(seed)
    m = torch.nn.Sequential(torch.nn.Linear(64, 128), torch.nn.Tanh(), torch.nn.Linear(128, 10))
    return m.cuda()


def _train(model, opt, steps, first=1, evict=False):
    from bit_block_wise_gb300 import paged_prefetch
    for k in range(first, first + steps):
        g = torch.Generator(device="cuda")
        g.manual_seed(1000 + k)
        x = torch.randn(32, 64, generator=g, device="cuda")
        y = torch.randint(0, 10, (32,), generator=g, device="cuda")
        opt.zero_grad(set_to_none=True)
        torch.nn.functional.cross_entropy(model(x), y).backward()
        if evict:
            paged_prefetch([st.get(key) for st in opt.state.values()
                            for key in ("state1", "state2", "absmax1", "absmax2")], "cpu")
        opt.step()


@pytest.mark.parametrize("name", ["Adam8bit", "AdamW8bit", "Lion8bit", "AdEMAMix8bit"])
@pytest.mark.parametrize("prefetch", [True, False])
def test_paged_classes_equal_unpaged(bnb8, name, prefetch):
    from bit_block_wise_gb300 import optim as O
    m1 = _model(3)
    m2 = copy.deepcopy(m1)
    o1 = getattr(O, name)(m1.parameters(), manager=O.OptimManager())
    o2 = getattr(O, "Paged" + name)(m2.parameters(), manager=O.OptimManager(),
                                     page_prefetch=prefetch)
    assert o2.is_paged and not o1.is_paged
    _train(m1, o1, 4)
    _train(m2, o2, 4, evict=True)
    torch.cuda.synchronize()
    # the first step created every parameter's state: one paged buffer
    bufs = {t.untyped_storage().data_ptr() for st in o2.state.values() for t in st.values()
            if torch.is_tensor(t)}
    assert len(bufs) == 1
    for a, b in zip(m1.parameters(), m2.parameters()):
        assert torch.equal(a, b)
    for a, b in zip(m1.parameters(), m2.parameters()):
        for key, val in o1.state[a].items():
            assert torch.equal(val, o2.state[b][key]) if torch.is_tensor(val) else val == o2.state[b][key]


def test_paged_state_dict_round_trip(bnb8):
    from bit_block_wise_gb300 import optim as O
    m1 = _model(4)
    o1 = O.PagedAdam8bit(m1.parameters(), manager=O.OptimManager())
    _train(m1, o1, 2)
    m2 = copy.deepcopy(m1)
    o2 = O.PagedAdam8bit(m2.parameters(), manager=O.OptimManager())
    o2.load_state_dict(copy.deepcopy(o1.state_dict()))
    for p in m2.parameters():
        for key in ("state1", "state2", "absmax1", "absmax2"):
            if key in o2.state[p]:
                bnb8.paged_prefetch(o2.state[p][key], "cpu")  # managed memory accepts it
    assert len({t.untyped_storage().data_ptr() for st in o2.state.values() for t in st.values()
                if torch.is_tensor(t)}) == 1
    _train(m1, o1, 2, first=3)
    _train(m2, o2, 2, first=3)
    torch.cuda.synchronize()
    for a, b in zip(m1.parameters(), m2.parameters()):
        assert torch.equal(a, b)
