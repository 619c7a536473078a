"""The torch.optim-style wrapper (bit_block_wise_gb300.optim) on the GPU:
bit-identical to direct library calls, state_dict round trips that resume
bit for bit, per-parameter overrides."""
import copy
import io

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

CLASSES = ["Adam8bit", "AdamW8bit", "Momentum8bit", "RMSprop8bit", "Adagrad8bit", "Lion8bit",
           "AdEMAMix8bit"]


@pytest.fixture(scope="module")
def bnb8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_block_wise_gb300 as m
    m.lib()
    return m


def _model(dtype, seed):
    torch.manual_seed(seed)
    # 64x128 weight (8,192 elements): 8-bit state; the others stay below
    # min_8bit_size (4,096) and keep 32-bit state
    m = torch.nn.Sequential(torch.nn.Linear(64, 128), torch.nn.Tanh(), torch.nn.Linear(128, 10))
    return m.cuda().to(dtype)


def _batch(k, dtype):
    g = torch.Generator(device="cuda")
    g.manual_seed(1000 + k)
    x = torch.randn(32, 64, generator=g, device="cuda").to(dtype)
    y = torch.randint(0, 10, (32,), generator=g, device="cuda")
    return x, y


def _train(model, opt, steps, dtype, first=1):
    for k in range(first, first + steps):
        x, y = _batch(k, dtype)
        opt.zero_grad(set_to_none=True)
        torch.nn.functional.cross_entropy(model(x).float(), y).backward()
        opt.step()


@pytest.mark.parametrize("cls", CLASSES)
def test_wrapper_equals_direct_calls(bnb8, cls):
    from bit_block_wise_gb300 import optim as O
    m1 = _model(torch.float32, 1)
    m2 = copy.deepcopy(m1)
    opt = getattr(O, cls)(m1.parameters(), manager=O.OptimManager())
    name = opt.optim
    hpd = dict(opt.defaults)
    # the same updates through the library directly
    s, u = bnb8.bnb8_create_qmap(True).cuda(), bnb8.bnb8_create_qmap(False).cuda()
    q1, q2 = (u, None) if name in ("rmsprop", "adagrad") else (s, u if name in ("adam", "adamw", "ademamix") else None)
    states = {}
    for k in range(1, 5):
        x, y = _batch(k, torch.float32)
        opt.zero_grad(set_to_none=True)
        torch.nn.functional.cross_entropy(m1(x).float(), y).backward()
        opt.step()
        for p in m2.parameters():
            p.grad = None
        torch.nn.functional.cross_entropy(m2(x).float(), y).backward()
        plist = []
        for p in m2.parameters():
            if p not in states:
                bits = 8 if p.numel() >= 4096 else 32
                states[p] = (*bnb8.zero_state(p.data, name, bits, 256), bits)
            s1, s2, a1, a2, bits = states[p]
            plist.append(bnb8.ParamState(p.data, p.grad, s1, s2, a1, a2, bits))
        betas = hpd["betas"]
        bnb8.step(plist, bnb8.HParams(optim=name, lr=hpd["lr"], beta1=betas[0], beta2=betas[1],
                                      beta3=betas[2] if len(betas) > 2 else 0.9999,
                                      alpha=hpd["alpha"], eps=hpd["eps"],
                                      weight_decay=hpd["weight_decay"], step=k), q1, q2)
    torch.cuda.synchronize()
    for a, b in zip(m1.parameters(), m2.parameters()):
        assert torch.equal(a, b)
    for p1, p2 in zip(m1.parameters(), m2.parameters()):
        st = opt.state[p1]
        assert torch.equal(st["state1"], states[p2][0])
        assert st["state_bits"] == states[p2][4]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("cls", ["Adam8bit", "AdEMAMix8bit"])
def test_state_dict_round_trip_resumes_bit_for_bit(bnb8, cls, dtype):
    from bit_block_wise_gb300 import optim as O
    straight = _model(dtype, 2)
    opt_s = getattr(O, cls)(straight.parameters(), manager=O.OptimManager())
    _train(straight, opt_s, 3, dtype)
    buf = io.BytesIO()
    torch.save({"model": straight.state_dict(), "opt": opt_s.state_dict()}, buf)
    _train(straight, opt_s, 3, dtype, first=4)

    buf.seek(0)
    ck = torch.load(buf, weights_only=False)
    resumed = _model(dtype, 99)
    resumed.load_state_dict(ck["model"])
    opt_r = getattr(O, cls)(resumed.parameters(), manager=O.OptimManager())
    opt_r.load_state_dict(ck["opt"])
    for p in resumed.parameters():
        st = opt_r.state[p]
        if st["state_bits"] == 8:
            assert st["state1"].dtype == torch.uint8
        if "absmax1" in st:
            assert st["absmax1"].dtype == torch.float32
        if st["state_bits"] == 32:
            assert st["state1"].dtype == torch.float32
    _train(resumed, opt_r, 3, dtype, first=4)
    torch.cuda.synchronize()
    for a, b in zip(straight.parameters(), resumed.parameters()):
        assert torch.equal(a, b)
    for a, b in zip(straight.parameters(), resumed.parameters()):
        for key in ("state1", "state2", "absmax1", "absmax2"):
            if key in opt_s.state[a]:
                assert torch.equal(opt_s.state[a][key], opt_r.state[b][key]), key


def test_override_config_per_parameter(bnb8):
    from bit_block_wise_gb300 import optim as O
    mgr = O.OptimManager()
    m = _model(torch.float32, 3)
    w = m[0].weight
    mgr.override_config(w, "optim_bits", 32)
    mgr.override_config(m[2].weight, key_value_dict={"lr": 0.0})
    before = m[2].weight.detach().clone()
    opt = O.Adam8bit(m.parameters(), manager=mgr)
    _train(m, opt, 2, torch.float32)
    torch.cuda.synchronize()
    assert opt.state[w]["state_bits"] == 32 and opt.state[w]["state1"].dtype == torch.float32
    assert torch.equal(m[2].weight, before)          # lr 0 for that weight
    assert not torch.equal(m[0].bias, _model(torch.float32, 3)[0].bias)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_carry_pnorm_matches_the_plain_pre_pass(bnb8, dtype):
    # AdamW (decoupled decay): the states never see p, so carrying ||p|| may
    # change p only through the multiplier's last bits (a different summation
    # order of the same binary32 partials)
    from bit_block_wise_gb300 import optim as O
    plain = _model(dtype, 5)
    carried = copy.deepcopy(plain)
    kw = dict(max_unorm=0.02, weight_decay=1e-2, manager=O.OptimManager())
    opt_p = O.AdamW8bit(plain.parameters(), **kw)
    opt_c = O.AdamW8bit(carried.parameters(), carry_pnorm=True, **kw)
    _train(plain, opt_p, 5, dtype)
    _train(carried, opt_c, 5, dtype)
    torch.cuda.synchronize()
    assert len(opt_c._carry_ws) >= 1 and len(opt_p._carry_ws) == 0
    for ws in opt_c._carry_ws.values():
        assert int(ws[:8].view(torch.int64).item()) != 0     # a step left its stamp
    tol = 1e-6 if dtype == torch.float32 else 2.0 ** -7
    for a, b in zip(plain.parameters(), carried.parameters()):
        assert torch.allclose(a.float(), b.float(), rtol=tol, atol=0.0)
        for key in ("state1", "state2", "absmax1", "absmax2"):
            if key in opt_p.state[a]:
                assert torch.equal(opt_p.state[a][key], opt_c.state[b][key]), key
    opt_c.load_state_dict(opt_c.state_dict())
    assert len(opt_c._carry_ws) == 0
