"""GPU parity at the full workload sizes, in the launch configuration that
bench.py times (one library call per step over the whole tensor list).

The oracle cannot step hundreds of millions of elements in seconds, but
blocks are independent: the oracle steps a sample of blocks (first, last and
random ones), with the state the GPU started from, and the GPU's result at
those blocks must equal it.  With max_unorm the oracle supplies its own
multiplier, computed over the whole tensor.  Properties that hold at any size
(untouched all-zero-gradient blocks under skip_zeros) are checked on every
block.
"""
import numpy as np
import pytest

import oracle
import workloads
from parity_util import (assert_same, gather, gather_absmax, maps, sample_blocks, to_dev,
                         to_host)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

S, U = maps()
TDT = {"f32": "float32", "bf16": "bfloat16", "f16": "float16"}


@pytest.fixture(scope="module")
def bnb8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_block_wise_gb300 as m
    m.lib()
    return m


def _maps_for(optim):
    if optim in ("adam", "adamw", "ademamix"):
        return S, U
    if optim in ("rmsprop", "adagrad"):
        return U, None
    return S, None


def _random_device_state(bnb8, optim, n, B, seed, dev):
    k = {"adam": 2, "adamw": 2, "ademamix": 3}.get(optim, 1)
    m = 2 if optim == "ademamix" else 1
    nb = (n + B - 1) // B
    s1 = workloads.torch_random_codes(n * m, seed, dev)
    a1 = workloads.torch_random_absmax(nb * m, 1e-3, seed + 1, dev)
    s2 = a2 = None
    if k >= 2:
        s2 = workloads.torch_random_codes(n, seed + 2, dev)
        a2 = workloads.torch_random_absmax(nb, 1e-6, seed + 3, dev)
    return s1, s2, a1, a2


def _sampled_oracle_state(ps, optim, n, B, blocks, dtype):
    """Host copy of the sampled blocks of one device tensor, laid out as a
    stand-alone tensor for the oracle."""
    nb = (n + B - 1) // B
    p = gather(ps.p, blocks, B, n)
    if optim == "ademamix":
        s1 = np.concatenate([gather(ps.s1, blocks, B, n, 0), gather(ps.s1, blocks, B, n, n)])
        a1 = np.concatenate([gather_absmax(ps.absmax1, blocks, nb, 0),
                             gather_absmax(ps.absmax1, blocks, nb, nb)])
    else:
        s1 = gather(ps.s1, blocks, B, n)
        a1 = gather_absmax(ps.absmax1, blocks, nb)
    s2 = a2 = None
    if ps.s2 is not None:
        s2 = gather(ps.s2, blocks, B, n)
        a2 = gather_absmax(ps.absmax2, blocks, nb)
    return oracle.TensorState(p, s1, s2, a1, a2, 8)


def _check_sampled(bnb8, ps, before, g_host, optim, dtype, n, B, blocks, hp, clip=None,
                   p_tol=False, tag=""):
    q1, q2 = _maps_for(optim)
    # the last block may be partial: step it on its own so that every
    # oracle tensor has whole blocks except possibly its end
    full = [b for b in blocks if (b + 1) * B <= n]
    part = [b for b in blocks if (b + 1) * B > n]
    after = _sampled_oracle_state(ps, optim, n, B, blocks, dtype)
    for group in (full, part):
        if not group:
            continue
        ref = _subset(before, optim, B, n, blocks, group)
        got = _subset(after, optim, B, n, blocks, group)
        g = _subset_array(g_host, B, n, blocks, group)
        oracle.step(oracle.HParams(optim=optim, **hp), ref, g, dtype, B, q1, q2, clip=clip)
        if p_tol:
            a = oracle.to_f32(got.p, dtype).astype(np.float64)
            b = oracle.to_f32(ref.p, dtype).astype(np.float64)
            if dtype == "f32":
                np.testing.assert_allclose(a, b, rtol=1e-6, atol=1e-12, err_msg=tag)
            else:
                ulp = np.abs(b) * (2.0 ** -7 if dtype == "bf16" else 2.0 ** -10)
                assert np.all(np.abs(a - b) <= ulp + 1e-30), tag
        else:
            assert_same(tag + " p", got.p, ref.p)
        assert_same(tag + " s1", got.s1, ref.s1)
        assert_same(tag + " s2", got.s2, ref.s2)
        assert_same(tag + " absmax1", got.absmax1, ref.absmax1)
        assert_same(tag + " absmax2", got.absmax2, ref.absmax2)


def _block_slices(B, n, blocks, group):
    out, pos = [], 0
    for b in blocks:
        ln = min(n, (b + 1) * B) - b * B
        if b in group:
            out.append((pos, pos + ln))
        pos += ln
    return out, pos


def _subset_array(a, B, n, blocks, group):
    sl, _ = _block_slices(B, n, blocks, group)
    return np.concatenate([a[lo:hi] for lo, hi in sl])


def _subset(t, optim, B, n, blocks, group):
    sl, total = _block_slices(B, n, blocks, group)
    cut = lambda a, off=0: np.concatenate([a[off + lo:off + hi] for lo, hi in sl])
    bidx = [blocks.index(b) for b in group]
    nbs = len(blocks)
    if optim == "ademamix":
        s1 = np.concatenate([cut(t.s1), cut(t.s1, total)])
        a1 = np.concatenate([t.absmax1[bidx], t.absmax1[[nbs + i for i in bidx]]])
    else:
        s1 = cut(t.s1)
        a1 = t.absmax1[bidx]
    s2 = None if t.s2 is None else cut(t.s2)
    a2 = None if t.absmax2 is None else t.absmax2[bidx]
    return oracle.TensorState(cut(t.p).copy(), s1.copy(), None if s2 is None else s2.copy(),
                              a1.copy(), None if a2 is None else a2.copy(), 8)


def _single_tensor_case(bnb8, optim, dtype, n, B, hp, grad, seed, steps=2, nsample=48,
                        rows=None):
    dev = torch.device("cuda")
    tdt = getattr(torch, TDT[dtype])
    p = workloads.torch_normal(n, 0.02, seed, dev, tdt)
    s1, s2, a1, a2 = _random_device_state(bnb8, optim, n, B, seed + 1, dev)
    ps = bnb8.ParamState(p, None, s1, s2, a1, a2, 8)
    q1, q2 = _maps_for(optim)
    qd1, qd2 = to_dev(q1), None if q2 is None else to_dev(q2)
    blocks = sample_blocks(n, B, nsample, seed)
    for k in range(1, steps + 1):
        g = grad(k)
        ps.g = g
        before = _sampled_oracle_state(ps, optim, n, B, blocks, dtype)
        g_host = gather(g, blocks, B, n)
        zero_blocks = None
        if hp.get("skip_zeros"):
            nbf = n // B
            zero_blocks = (g[: nbf * B].view(nbf, B) == 0).all(dim=1)
            keep = (ps.p.clone(), ps.s1.clone(), ps.absmax1.clone())
        bnb8.step([ps], bnb8.HParams(optim=optim, blocksize=B, step=k, **hp), qd1, qd2)
        torch.cuda.synchronize()
        _check_sampled(bnb8, ps, before, g_host, optim, dtype, n, B, blocks, dict(hp, step=k),
                       tag=f"{optim}/{dtype}/n={n}/B{B}/step{k}")
        if zero_blocks is not None:
            # every all-zero-gradient block keeps p, codes and absmax bit-identical
            assert bool(zero_blocks.any())
            idx = zero_blocks.nonzero().squeeze(1)
            pv, cv, av = keep
            nbf = n // B
            assert torch.equal(ps.p[: nbf * B].view(nbf, B)[idx].view(torch.int16 if dtype != "f32" else torch.int32),
                               pv[: nbf * B].view(nbf, B)[idx].view(torch.int16 if dtype != "f32" else torch.int32))
            assert torch.equal(ps.s1[: nbf * B].view(nbf, B)[idx], cv[: nbf * B].view(nbf, B)[idx])
            assert torch.equal(ps.absmax1[idx].view(torch.int32), av[idx].view(torch.int32))


@pytest.mark.parametrize("optim,B", [("adam", 256), ("adamw", 256), ("adam", 2048)])
def test_adam_4096x4096_f32(bnb8, optim, B):
    n = 4096 * 4096
    dev = torch.device("cuda")
    grad = lambda k: workloads.torch_normal_with_outliers(n, 1e-3, 1e-1, 0.01, 500 + k, dev)
    _single_tensor_case(bnb8, optim, "f32", n, B,
                        dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=1e-2),
                        grad, seed=11)


ONE_STATE = {"momentum": dict(lr=0.01, beta1=0.9), "rmsprop": dict(lr=0.01, beta1=0.9),
             "adagrad": dict(lr=0.01), "lion": dict(lr=1e-4, beta1=0.9, beta2=0.99)}


@pytest.mark.parametrize("optim", sorted(ONE_STATE))
@pytest.mark.parametrize("skip", [True, False])
def test_one_state_embedding_rows_bf16(bnb8, optim, skip):
    rows, cols = 50257, 1024
    n = rows * cols
    dev = torch.device("cuda")
    grad = lambda k: workloads.torch_sparse_rows(rows, cols, 0.1, 1e-3, 600 + k, dev,
                                                 torch.bfloat16)
    _single_tensor_case(bnb8, optim, "bf16", n, 256,
                        dict(ONE_STATE[optim], weight_decay=1e-2, skip_zeros=skip), grad,
                        seed=21)


@pytest.mark.parametrize("optim", sorted(ONE_STATE))
def test_one_state_dense_64m_bf16(bnb8, optim):
    n = 1 << 26
    dev = torch.device("cuda")
    grad = lambda k: workloads.torch_normal(n, 1e-3, 700 + k, dev, torch.bfloat16)
    _single_tensor_case(bnb8, optim, "bf16", n, 256, dict(ONE_STATE[optim]), grad, seed=31,
                        steps=1)


def test_ademamix_64m_f32(bnb8):
    n = 1 << 26
    dev = torch.device("cuda")
    grad = lambda k: workloads.torch_normal(n, 1e-3, 800 + k, dev)
    _single_tensor_case(bnb8, "ademamix", "f32", n, 256,
                        dict(lr=1e-3, beta1=0.9, beta2=0.999, beta3=0.9999, alpha=5.0,
                             t_alpha=100, t_beta3=100, eps=1e-8), grad, seed=41)


def test_gpt2xl_list_bf16_max_unorm(bnb8):
    """One step over the 580-tensor GPT-2-XL-shaped list (1.56 G elements),
    small tensors at 32-bit state, max_unorm 1.0, wd 0.1."""
    dev = torch.device("cuda")
    B = 256
    shapes = workloads.gpt2_xl_params()
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1, max_unorm=1.0,
              step=3)
    params = []
    for i, (name, n) in enumerate(shapes):
        p = workloads.torch_normal(n, 0.02, 9000 + i, dev, torch.bfloat16)
        g = workloads.torch_normal(n, 1e-3, 19000 + i, dev, torch.bfloat16)
        if n >= 4096:
            s1, s2, a1, a2 = _random_device_state(bnb8, "adam", n, B, 29000 + 10 * i, dev)
            params.append(bnb8.ParamState(p, g, s1, s2, a1, a2, 8))
        else:
            s1 = workloads.torch_normal(n, 1e-3, 39000 + i, dev)
            s2 = workloads.torch_normal(n, 1e-6, 49000 + i, dev).abs_()
            params.append(bnb8.ParamState(p, g, s1, s2, None, None, 32))
    names = [nm for nm, _ in shapes]
    check = ["wte", "wpe", "h0.attn.c_attn.weight", "h0.attn.c_attn.bias", "h23.mlp.c_fc.weight",
             "h47.mlp.c_proj.weight", "h5.ln_1.weight", "h10.attn.c_proj.bias", "ln_f.bias"]
    saved = {}
    for nm in check:
        ps = params[names.index(nm)]
        saved[nm] = dict(p=to_host(ps.p), g=to_host(ps.g), s1=to_host(ps.s1), s2=to_host(ps.s2),
                         a1=to_host(ps.absmax1), a2=to_host(ps.absmax2))
    bnb8.step(params, bnb8.HParams(optim="adam", blocksize=B, **hp), to_dev(S), to_dev(U))
    torch.cuda.synchronize()
    for nm in check:
        ps = params[names.index(nm)]
        sv = saved[nm]
        n = ps.p.numel()
        bits = ps.state_bits
        ref = oracle.TensorState(sv["p"].copy(), sv["s1"].copy(), sv["s2"].copy(),
                                 None if sv["a1"] is None else sv["a1"].copy(),
                                 None if sv["a2"] is None else sv["a2"].copy(), bits)
        ohp = oracle.HParams(optim="adam", **hp)
        clip, _, _ = oracle.unorm_scale(ohp, ref, sv["g"], "bf16", B, S, U)
        assert clip < 1.0, nm
        if bits == 32 or n <= 64 * B:
            oracle.step(ohp, ref, sv["g"], "bf16", B, S, U, clip=clip)
            got = oracle.TensorState(to_host(ps.p), to_host(ps.s1), to_host(ps.s2),
                                     to_host(ps.absmax1), to_host(ps.absmax2), bits)
            a = oracle.to_f32(got.p, "bf16").astype(np.float64)
            b = oracle.to_f32(ref.p, "bf16").astype(np.float64)
            assert np.all(np.abs(a - b) <= np.abs(b) * 2.0 ** -7 + 1e-30), nm
            for x, y, lab in ((got.s1, ref.s1, "s1"), (got.s2, ref.s2, "s2"),
                              (got.absmax1, ref.absmax1, "a1"), (got.absmax2, ref.absmax2, "a2")):
                if y is not None:
                    assert_same(f"{nm} {lab}", x, y)
        else:
            blocks = sample_blocks(n, B, 40, hash(nm) % 1000)
            before = _subset_from_host(sv, blocks, B, n)
            g_host = _concat_blocks(sv["g"], blocks, B, n)
            _check_sampled(bnb8, ps, before, g_host, "adam", "bf16", n, B, blocks,
                           dict(hp), clip=clip, p_tol=True, tag=nm)


def _concat_blocks(a, blocks, B, n):
    return np.concatenate([a[b * B:min(n, (b + 1) * B)] for b in blocks])


def _subset_from_host(sv, blocks, B, n):
    return oracle.TensorState(_concat_blocks(sv["p"], blocks, B, n),
                              _concat_blocks(sv["s1"], blocks, B, n),
                              _concat_blocks(sv["s2"], blocks, B, n),
                              sv["a1"][blocks].copy(), sv["a2"][blocks].copy(), 8)
