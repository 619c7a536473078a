"""The torch.optim-style wrapper on the host: which parameters get 8-bit
state, what the zero state holds, config overrides (no GPU needed)."""
import pytest
import torch

from bit_block_wise_gb300 import optim as O


def _params():
    return [torch.nn.Parameter(torch.zeros(8192)), torch.nn.Parameter(torch.zeros(100)),
            torch.nn.Parameter(torch.zeros(5000))]


def test_min_8bit_size_and_overrides():
    mgr = O.OptimManager()
    ps = _params()
    mgr.override_config(ps[2], "optim_bits", 32)
    opt = O.Adam8bit(ps, manager=mgr)
    g = opt.param_groups[0]
    opt._init_states([(p, opt._config(g, p)) for p in ps])
    st = [opt.state[p] for p in ps]
    assert [s["state_bits"] for s in st] == [8, 32, 32]
    assert st[0]["state1"].dtype == torch.uint8 and st[0]["absmax1"].numel() == 8192 // 256
    assert torch.all(st[0]["state1"] == 127)          # the signed map's 0.0
    assert torch.all(st[0]["state2"] == 0)            # the unsigned map's 0.0
    assert st[1]["state1"].dtype == torch.float32 and "absmax1" not in st[1]


def test_tensorwise_state_has_one_absmax_per_state():
    opt = O.AdEMAMix8bit(_params()[:1], blocksize=0, manager=O.OptimManager())
    p = opt.param_groups[0]["params"][0]
    opt._init_states([(p, opt._config(opt.param_groups[0], p))])
    st = opt.state[p]
    assert st["absmax1"].numel() == 2 and st["absmax2"].numel() == 1
    assert st["state1"].numel() == 2 * p.numel()


def test_config_errors():
    with pytest.raises(ValueError):
        O.OptimManager().override_config(_params()[0], "no_such_key", 1)
    with pytest.raises(ValueError):
        O.Optimizer8bit(_params(), optim="sgd")
    with pytest.raises(ValueError):
        O.Adam8bit(_params(), optim_bits=16)


def test_paged_classes():
    for name in ("Adam8bit", "AdamW8bit", "Lion8bit", "AdEMAMix8bit"):
        paged = getattr(O, "Paged" + name)(_params(), manager=O.OptimManager())
        plain = getattr(O, name)(_params(), manager=O.OptimManager())
        assert paged.is_paged and paged.page_prefetch and not plain.is_paged
        assert paged.optim == plain.optim and paged.defaults == plain.defaults
    assert not O.PagedAdam8bit(_params(), page_prefetch=False).page_prefetch
