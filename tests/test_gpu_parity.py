"""GPU parity: the CUDA library (called through its C ABI via the binding)
against the CPU oracle, element by element, on seeded inputs.

Bar: codes and absmax bit-exact; parameters bit-exact too (the kernels run
the oracle's binary32 operation sequence: IEEE division and square root,
fused multiply-adds exactly where the update's definition has them and no
other contraction), except where max_unorm's norms are summed in a different
order: there the step multiplier matches to about 1e-6 relative, so p is
within 1e-6 of |p| plus 1e-6 of the update's size (binary32) / 1 ulp
(16-bit).
"""
import numpy as np
import pytest

import oracle
import workloads
from parity_util import assert_same, map_pair, maps, random_state, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

S, U = maps()
OPTIMS = ["adam", "adamw", "momentum", "rmsprop", "adagrad", "lion", "ademamix"]
HP_BASE = {
    "adam": dict(lr=1e-3, beta1=0.9, beta2=0.999),
    "adamw": dict(lr=1e-3, beta1=0.9, beta2=0.999),
    "momentum": dict(lr=0.01, beta1=0.9),
    "rmsprop": dict(lr=0.01, beta1=0.9),
    "adagrad": dict(lr=0.01),
    "lion": dict(lr=1e-4, beta1=0.9, beta2=0.99),
    "ademamix": dict(lr=1e-3, beta1=0.9, beta2=0.999, beta3=0.9999, alpha=5.0, t_alpha=10,
                     t_beta3=10),
}


@pytest.fixture(scope="module")
def bnb8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_block_wise_gb300 as m
    m.lib()
    return m


@pytest.fixture(scope="module")
def qdev(bnb8):
    return to_dev(S), to_dev(U)


def _host_to(x, dtype):
    return oracle.to_storage(x, dtype)


def run_case(bnb8, qdev, optim, dtype, bits, B, sizes, steps=3, skip_zeros=False, wd=0.0,
             gscale=1.0, max_unorm=0.0, zero_frac=0.0, seed=0, init="random", extra_hp=None,
             offsets=None, neg_zero=False):
    """Run `steps` updates of a tensor list on the GPU and on the oracle and
    compare after every step.  B = 0: tensor-wise quantization (the oracle
    takes each tensor as one block)."""
    q1, q2 = map_pair(optim, S, U)
    qd1 = qdev[0] if q1 is S else qdev[1]
    qd2 = None if q2 is None else qdev[1]
    refs, params, keep = [], [], []
    for i, n in enumerate(sizes):
        p = _host_to(workloads.normal(n, 0.1, seed + 10 * i), dtype)
        b = bits[i] if isinstance(bits, (list, tuple)) else bits
        Bo = B or n
        if init == "zero":
            st = oracle.zero_state(optim, n, b, Bo, q1, q2)
        else:
            st = random_state(optim, n, b, Bo, seed + 10 * i + 1, q1, q2)
        refs.append(oracle.TensorState(p.copy(), *[None if a is None else a.copy() for a in st], b))
        dev = [to_dev(p, dtype)] + [to_dev(a) for a in st]
        if offsets is not None and offsets[i]:
            # misaligned storage: same values at an element offset (scalar path)
            off = offsets[i]
            shifted = []
            for t in dev:
                if t is None:
                    shifted.append(None)
                    continue
                buf = torch.empty(t.numel() + off, dtype=t.dtype, device=t.device)
                buf[off:].copy_(t)
                keep.append(buf)
                shifted.append(buf[off:])
            dev = shifted
        params.append(bnb8.ParamState(dev[0], None, dev[1], dev[2], dev[3], dev[4], b))
    for k in range(1, steps + 1):
        hp = dict(HP_BASE[optim])
        hp.update(extra_hp or {})
        hp.update(weight_decay=wd, gnorm_scale=gscale, max_unorm=max_unorm, step=k,
                  skip_zeros=skip_zeros)
        ghost = []
        for i, n in enumerate(sizes):
            g = workloads.normal(n, 1e-2, seed + 1000 * k + i)
            if zero_frac:
                rng = np.random.default_rng(seed + 7 * k + i)
                g[rng.random(n) < zero_frac] = 0.0
                # whole zero blocks too
                Bz = B or 256
                nb = (n + Bz - 1) // Bz
                for blk in rng.choice(nb, size=max(1, nb // 3), replace=False):
                    g[blk * Bz:(blk + 1) * Bz] = 0.0
                if neg_zero:
                    g[(g == 0.0) & (rng.random(n) < 0.5)] = -0.0
            g = _host_to(g, dtype)
            ghost.append(g)
            gd = to_dev(g, dtype)
            if offsets is not None and offsets[i]:
                buf = torch.empty(gd.numel() + offsets[i], dtype=gd.dtype, device=gd.device)
                buf[offsets[i]:].copy_(gd)
                keep.append(buf)
                gd = buf[offsets[i]:]
            params[i].g = gd
        bnb8.step(params, bnb8.HParams(optim=optim, blocksize=B, **hp), qd1, qd2)
        ohp = oracle.HParams(optim=optim, **hp)
        before = [oracle.to_f32(r.p, dtype).astype(np.float64) for r in refs]
        for i, n in enumerate(sizes):
            oracle.step(ohp, refs[i], ghost[i], dtype, B or n, q1, q2)
        torch.cuda.synchronize()
        for i, (ps, r) in enumerate(zip(params, refs)):
            tag = f"{optim}/{dtype}/bits{r.state_bits}/B{B}/step{k}/t{i}(n={sizes[i]})"
            if max_unorm > 0:
                got = oracle.to_f32(to_host(ps.p), dtype).astype(np.float64)
                want = oracle.to_f32(r.p, dtype).astype(np.float64)
                if dtype == "f32":
                    # the multiplier matches to about 1e-6 relative, so p does
                    # to 1e-6 of |p| plus 1e-6 of the update (an update that
                    # nearly cancels p leaves |p| no scale of its own)
                    tol = 1e-6 * (np.abs(want) + np.abs(want - before[i])) + 1e-12
                    bad = np.abs(got - want) > tol
                    assert not bad.any(), (tag, np.flatnonzero(bad)[:5], got[bad][:5], want[bad][:5])
                else:
                    # one unit in the last place of the 16-bit format
                    ulp = np.abs(want) * (2.0 ** -7 if dtype == "bf16" else 2.0 ** -10)
                    assert np.all(np.abs(got - want) <= ulp + 1e-30), tag
                # continue from identical parameters so the check stays per step
                ps.p.copy_(to_dev(r.p, dtype))
            else:
                assert_same(tag + " p", to_host(ps.p), r.p)
            assert_same(tag + " s1", to_host(ps.s1), r.s1)
            assert_same(tag + " s2", to_host(ps.s2), r.s2)
            assert_same(tag + " absmax1", to_host(ps.absmax1), r.absmax1)
            assert_same(tag + " absmax2", to_host(ps.absmax2), r.absmax2)
    return params, refs


# ---------------------------------------------------------------------------
# quantize / dequantize
# ---------------------------------------------------------------------------

def _special_values(n, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(n).astype(np.float32) * np.float32(0.01)
    x[::7] = 0.0
    x[1::11] = -0.0
    x[2::13] = np.float32(1e-30) * rng.standard_normal(x[2::13].size).astype(np.float32)
    x[3::17] = np.float32(3e-39)                                   # subnormal
    x[4::19] = rng.choice(S, x[4::19].size) * np.float32(0.01)     # exact levels
    return x


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("B", [64, 128, 256, 512, 1024, 2048, 4096])
@pytest.mark.parametrize("signed", [True, False])
def test_quantize_matches_oracle(bnb8, dtype, B, signed):
    q = S if signed else U
    n = 5 * B + 77
    x = _host_to(_special_values(n, B), dtype)
    x_dev = to_dev(x, dtype)
    codes, absmax = bnb8.bnb8_quantize_blockwise(x_dev, to_dev(q), B)
    oc, oa = oracle.quantize_blockwise(x, dtype, q, B)
    torch.cuda.synchronize()
    assert_same("codes", to_host(codes), oc)
    assert_same("absmax", to_host(absmax), oa)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("B", [64, 256, 4096])
def test_dequantize_matches_oracle(bnb8, dtype, B):
    n = 3 * B + 5
    codes = workloads.random_codes(n, B)
    absmax = workloads.random_absmax((n + B - 1) // B, 2.0, B + 1)
    out = bnb8.bnb8_dequantize_blockwise(to_dev(codes), to_dev(absmax), to_dev(S), B,
                                         dtype={"f32": torch.float32, "bf16": torch.bfloat16,
                                                "f16": torch.float16}[dtype])
    torch.cuda.synchronize()
    assert_same("dequant", to_host(out), oracle.dequantize_blockwise(codes, absmax, S, B, dtype))


def test_quantize_degenerate_blocks(bnb8):
    # all-zero block, a block of subnormals whose reciprocal overflows, a
    # block at the binary32 maximum, and exact map levels at power-of-two scale
    B = 256
    blocks = [np.zeros(B, np.float32),
              np.full(B, np.float32(1e-45)) * np.sign(np.random.default_rng(0).standard_normal(B)).astype(np.float32),
              np.linspace(-3.4e38, 3.4e38, B).astype(np.float32),
              (S * np.float32(2.0 ** -20)).astype(np.float32)]
    x = np.concatenate(blocks).astype(np.float32)
    for q in (S, U):
        codes, absmax = bnb8.bnb8_quantize_blockwise(to_dev(x), to_dev(q), B)
        oc, oa = oracle.quantize_blockwise(x, "f32", q, B)
        torch.cuda.synchronize()
        assert_same("codes", to_host(codes), oc)
        assert_same("absmax", to_host(absmax), oa)


def test_quantize_fallback_map(bnb8):
    # a map with two midpoints inside one search bucket (levels 1e-3 and
    # 1.0001e-3) and one in the tiny bucket: the kernels must take the exact
    # binary-search path and still match the oracle
    q = np.sort(np.concatenate([np.linspace(-1, 1, 250), [1e-3, 1.0001e-3, 1.0002e-3, 1e-9,
                                                          2e-9, 3e-9]]).astype(np.float32))
    assert q.size == 256 and np.all(np.diff(q) > 0)
    x = _special_values(4 * 256 + 9, 5)
    x[100:140] = np.float32(1.00005e-3) * 0.01
    codes, absmax = bnb8.bnb8_quantize_blockwise(to_dev(x), to_dev(q), 256)
    oc, oa = oracle.quantize_blockwise(x, "f32", q, 256)
    torch.cuda.synchronize()
    assert_same("codes", to_host(codes), oc)
    assert_same("absmax", to_host(absmax), oa)


# ---------------------------------------------------------------------------
# optimizer steps
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("optim", OPTIMS)
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("bits", [8, 32])
def test_step_matches_oracle(bnb8, qdev, optim, dtype, bits):
    # several tiles, a ragged tail block, a single-element tensor
    run_case(bnb8, qdev, optim, dtype, bits, 256, [7 * 256 + 77, 4096, 1], steps=3,
             wd=1e-2, seed=1)


@pytest.mark.parametrize("optim", OPTIMS)
@pytest.mark.parametrize("B", [64, 128, 512, 2048, 4096])
def test_step_blocksizes(bnb8, qdev, optim, B):
    run_case(bnb8, qdev, optim, "f32", 8, B, [3 * B + 5, B], steps=2, seed=2)


@pytest.mark.parametrize("optim", OPTIMS)
@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_step_from_zero_state(bnb8, qdev, optim, dtype):
    run_case(bnb8, qdev, optim, dtype, 8, 256, [5000], steps=5, init="zero", seed=3)


@pytest.mark.parametrize("optim", OPTIMS)
@pytest.mark.parametrize("bits", [8, 32])
@pytest.mark.parametrize("B", [256, 2048])
def test_step_skip_zeros(bnb8, qdev, optim, bits, B):
    run_case(bnb8, qdev, optim, "bf16", bits, B, [6 * B + 3], steps=3, skip_zeros=True,
             zero_frac=0.2, wd=1e-2, seed=4)


@pytest.mark.parametrize("optim", OPTIMS)
@pytest.mark.parametrize("bits", [8, 32])
@pytest.mark.parametrize("init", ["zero", "random"])
def test_step_zero_gradients_not_skipped(bnb8, qdev, optim, bits, init):
    """Zero gradients (+0 and -0) with skip_zeros off and no decay: from a zero
    state the second moments stay exactly 0 (sqrt(0) + eps), and zero
    numerators reach the division (0 / d)."""
    run_case(bnb8, qdev, optim, "bf16", bits, 256, [6 * 256 + 3, 1000], steps=3, zero_frac=0.3,
             init=init, seed=44, neg_zero=True)


@pytest.mark.parametrize("optim", OPTIMS)
def test_step_gnorm_scale_and_coupled_decay(bnb8, qdev, optim):
    run_case(bnb8, qdev, optim, "f32", 8, 256, [3000], steps=2, wd=0.1, gscale=0.37, seed=5)


@pytest.mark.parametrize("optim", OPTIMS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_step_max_unorm(bnb8, qdev, optim, dtype):
    run_case(bnb8, qdev, optim, dtype, [8, 32, 8], 256, [4000, 300, 256 * 9], steps=3,
             max_unorm=0.05, wd=1e-2, seed=6)


@pytest.mark.parametrize("optim", ["adam", "lion"])
@pytest.mark.parametrize("max_unorm", [0.0, 0.05])
def test_step_list_of_whole_and_ragged_tensors(bnb8, qdev, optim, max_unorm):
    # the planner launches whole-chunk tensors apart from the ragged ones and
    # 32-bit tensors apart from both: results and per-tensor multipliers must
    # not depend on that grouping
    sizes = [512 * 4, 1000, 512 * 9, 300, 777, 512 * 2, 256 * 3, 4096]
    bits = [8, 8, 8, 32, 8, 8, 8, 32]
    run_case(bnb8, qdev, optim, "f32", bits, 256, sizes, steps=2, max_unorm=max_unorm, wd=1e-2,
             seed=17)


@pytest.mark.parametrize("optim", ["adam", "momentum", "ademamix"])
@pytest.mark.parametrize("B", [256, 2048])
def test_unorm_scales_match_oracle(bnb8, qdev, optim, B):
    # B = 2048: the pre-pass's two-pass shape (fp32, <= 2 states) or its
    # one-pass shape (AdEMAMix), four warps per block, a ragged last block
    q1, q2 = map_pair(optim, S, U)
    sizes, bits = [5000, 700, 256 * 40 + 3], [8, 32, 8]
    params, refs = [], []
    for i, n in enumerate(sizes):
        p = workloads.normal(n, 0.02, 70 + i)
        st = random_state(optim, n, bits[i], B, 80 + i, q1, q2)
        refs.append(oracle.TensorState(p.copy(), *st, bits[i]))
        params.append(bnb8.ParamState(to_dev(p), to_dev(workloads.normal(n, 1e-2, 90 + i)),
                                      *[to_dev(a) for a in st], bits[i]))
    hp = dict(HP_BASE[optim], max_unorm=0.02, step=4)
    qd1 = qdev[0] if q1 is S else qdev[1]
    scales = bnb8.bnb8_unorm(params, bnb8.HParams(optim=optim, blocksize=B, **hp), qd1,
                             None if q2 is None else qdev[1])
    torch.cuda.synchronize()
    got = to_host(scales)
    for i, (ps, r) in enumerate(zip(params, refs)):
        want, unorm, pnorm = oracle.unorm_scale(oracle.HParams(optim=optim, **hp), r,
                                                to_host(ps.g), "f32", B, q1, q2)
        assert abs(got[i] - want) <= 1e-6 * want, (i, got[i], want)
        assert got[i] < 1.0


def test_unorm_scales_chunked_sums(bnb8, qdev):
    # the per-tensor sums go through chunks of 512 blocks: a one-block
    # tensor, tensors whose last chunk is one block (the second one ragged)
    q1, q2 = S, U
    sizes = [100, 256 * 4097, 256 * 8192 + 5]
    params, refs = [], []
    for i, n in enumerate(sizes):
        p = workloads.normal(n, 0.02, 150 + i)
        st = random_state("adam", n, 8, 256, 160 + i, q1, q2)
        refs.append(oracle.TensorState(p.copy(), *st, 8))
        params.append(bnb8.ParamState(to_dev(p), to_dev(workloads.normal(n, 1e-2, 170 + i)),
                                      *[to_dev(a) for a in st], 8))
    hp = dict(HP_BASE["adam"], max_unorm=0.02, step=3)
    scales = bnb8.bnb8_unorm(params, bnb8.HParams(optim="adam", **hp), qdev[0], qdev[1])
    torch.cuda.synchronize()
    got = to_host(scales)
    for i, (ps, r) in enumerate(zip(params, refs)):
        want, _, _ = oracle.unorm_scale(oracle.HParams(optim="adam", **hp), r, to_host(ps.g),
                                        "f32", 256, q1, q2)
        assert abs(got[i] - want) <= 1e-6 * want, (i, got[i], want)
        assert got[i] < 1.0


def test_step_multi_tensor_list_over_launch_capacity(bnb8, qdev):
    # more tensors than one launch carries, mixed 8/32-bit, empty tensors
    rng = np.random.default_rng(9)
    sizes = [int(x) for x in rng.integers(1, 3000, 150)]
    sizes[5] = 0
    sizes[77] = 0
    bits = [8 if n >= 1024 else 32 for n in sizes]
    run_case(bnb8, qdev, "adam", "bf16", bits, 256, sizes, steps=2, seed=10)


@pytest.mark.parametrize("optim", ["adam", "ademamix", "lion"])
def test_step_unaligned_tensors(bnb8, qdev, optim):
    # element offsets that break 16-byte alignment: the scalar path
    run_case(bnb8, qdev, optim, "f32", 8, 256, [1000, 2049], steps=2, offsets=[1, 3], seed=11)
    run_case(bnb8, qdev, optim, "bf16", 32, 256, [1000, 2049], steps=2, offsets=[1, 3], seed=12)


def test_ademamix_ragged_m2_offset(bnb8, qdev):
    # n % 8 != 0 puts the m2 codes of s1 = [2, n] off the 8-byte grid
    run_case(bnb8, qdev, "ademamix", "f32", 8, 256, [1003, 517], steps=3, seed=13)


@pytest.mark.parametrize("optim", ["adam", "lion", "ademamix"])
@pytest.mark.parametrize("bits", [8, 32])
def test_split_blocks_pieces_equal_whole_tensor(bnb8, qdev, optim, bits):
    # blocks are independent: updating block-aligned views one by one is the
    # same update as updating the whole tensor (AdEMAMix 8-bit stays whole)
    q1, q2 = map_pair(optim, S, U)
    qd1 = qdev[0] if q1 is S else qdev[1]
    qd2 = None if q2 is None else qdev[1]
    n, B = 256 * 37 + 11, 256
    st = random_state(optim, n, bits, B, 400, q1, q2)
    p = workloads.normal(n, 0.1, 401)
    g = to_dev(workloads.normal(n, 1e-2, 402))
    whole = bnb8.ParamState(to_dev(p), g, *[to_dev(a) for a in st], bits)
    split = bnb8.ParamState(to_dev(p), g, *[to_dev(a) for a in st], bits)
    hp = bnb8.HParams(optim=optim, blocksize=B, step=2, weight_decay=1e-2, alpha=2.0)
    bnb8.step([whole], hp, qd1, qd2)
    _, pieces = bnb8.split_blocks(split, B, 5)
    for pc in pieces:
        bnb8.step([pc], hp, qd1, qd2)
    torch.cuda.synchronize()
    for name in ("p", "s1", "s2", "absmax1", "absmax2"):
        a, b = getattr(whole, name), getattr(split, name)
        if a is not None:
            assert_same(name, to_host(b), to_host(a))


# ---------------------------------------------------------------------------
# lists large enough that every CTA of the persistent grid visits many
# blocks: warps cross from one tensor into the next, ragged last blocks,
# tensors off the 16-byte grid next to aligned ones
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("optim,dtype", [("adam", "f32"), ("adamw", "bf16"), ("lion", "f32"),
                                         ("rmsprop", "f16"), ("ademamix", "f32")])
def test_step_many_blocks_per_cta(bnb8, qdev, optim, dtype):
    # 8,001 blocks of 256 elements: about 26 per CTA of 304, crossing tensors
    run_case(bnb8, qdev, optim, dtype, 8, 256, [256 * 5000 + 80, 256 * 3000], steps=2,
             wd=1e-2, seed=21)


@pytest.mark.parametrize("B", [64, 512, 4096])
def test_step_blocksizes_many_blocks_per_cta(bnb8, qdev, B):
    nblocks = 152 * (8192 // B) * 2 + 7
    run_case(bnb8, qdev, "adam", "f32", 8, B, [nblocks * B - 3, 5 * B], steps=2, seed=22)


def test_step_mixed_aligned_and_unaligned_tensors(bnb8, qdev):
    # the middle tensor starts off the 16-byte grid (scalar path) between two
    # aligned ones (vector path)
    sizes = [256 * 2000, 256 * 1500 + 9, 256 * 2500]
    run_case(bnb8, qdev, "adam", "f32", 8, 256, sizes, steps=2, offsets=[0, 1, 0], seed=23)


def test_step_ademamix_second_moment_offset_many_blocks(bnb8, qdev):
    # n % 16 != 0: m2's codes (n bytes into s1) are off the 16-byte grid
    run_case(bnb8, qdev, "ademamix", "bf16", 8, 256, [256 * 3000 + 8, 256 * 2000], steps=2,
             seed=24)


@pytest.mark.parametrize("optim", ["adam", "momentum", "ademamix"])
def test_stepper_equals_step(bnb8, qdev, optim):
    # arguments marshalled once, update number set per call: the same bits
    # as the plain entry point, step after step
    q1, q2 = map_pair(optim, S, U)
    qd1 = qdev[0] if q1 is S else qdev[1]
    qd2 = None if q2 is None else qdev[1]
    sizes = [256 * 300 + 5, 4096]
    a, b = [], []
    for i, n in enumerate(sizes):
        st = random_state(optim, n, 8, 256, 500 + i, q1, q2)
        p = workloads.normal(n, 0.1, 510 + i)
        g = to_dev(workloads.normal(n, 1e-2, 520 + i))
        a.append(bnb8.ParamState(to_dev(p), g, *[to_dev(x) for x in st], 8))
        b.append(bnb8.ParamState(to_dev(p), g, *[to_dev(x) for x in st], 8))
    hp = dict(HP_BASE[optim], weight_decay=1e-2)
    stepper = bnb8.Stepper(b, bnb8.HParams(optim=optim, step=1, **hp), qd1, qd2)
    for k in range(1, 4):
        bnb8.step(a, bnb8.HParams(optim=optim, step=k, **hp), qd1, qd2)
        stepper(k)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        for name in ("p", "s1", "s2", "absmax1", "absmax2"):
            if getattr(x, name) is not None:
                assert_same(name, to_host(getattr(y, name)), to_host(getattr(x, name)))


# ---------------------------------------------------------------------------
# maps other than the two dynamic maps: each kernel builds its search table
# from the map it is given, so new contents in the same buffer, and many
# different maps in a row, quantize exactly like the oracle
# ---------------------------------------------------------------------------

def _moved_levels(q, seed):
    """q with five interior levels moved between their neighbours: still an
    ascending map whose bucket search is exact, but a different table."""
    rng = np.random.default_rng(seed)
    q = q.copy()
    for _ in range(5):
        i = int(rng.integers(1, 255))
        q[i] = np.float32(q[i - 1] + (q[i + 1] - q[i - 1]) * np.float32(rng.uniform(0.2, 0.8)))
    return q


def test_quantize_map_rewritten_in_place(bnb8):
    x = _special_values(40 * 256 + 3, 31)
    qd = to_dev(S.copy())
    for k, q in enumerate([S, _moved_levels(S, 32), _moved_levels(S, 33), S]):
        qd.copy_(to_dev(q))
        codes, absmax = bnb8.bnb8_quantize_blockwise(to_dev(x), qd, 256)
        oc, oa = oracle.quantize_blockwise(x, "f32", q, 256)
        torch.cuda.synchronize()
        assert_same(f"codes/{k}", to_host(codes), oc)
        assert_same(f"absmax/{k}", to_host(absmax), oa)


def test_quantize_many_different_maps(bnb8):
    x = _special_values(9 * 256 + 100, 34)
    maps_dev = []
    for k in range(12):
        q = _moved_levels(U if k % 2 else S, 35 + k)
        qd = to_dev(q)
        maps_dev.append(qd)
        codes, absmax = bnb8.bnb8_quantize_blockwise(to_dev(x), qd, 128)
        oc, oa = oracle.quantize_blockwise(x, "f32", q, 128)
        torch.cuda.synchronize()
        assert_same(f"codes/{k}", to_host(codes), oc)
        assert_same(f"absmax/{k}", to_host(absmax), oa)


@pytest.mark.parametrize("optim", ["adam", "lion"])
def test_step_map_rewritten_in_place(bnb8, optim):
    # the second step runs with new contents in the same map buffers
    q1, q2 = map_pair(optim, S, U)
    n, B = 256 * 50 + 7, 256
    st = random_state(optim, n, 8, B, 40, q1, q2)
    p = workloads.normal(n, 0.1, 41)
    ref = oracle.TensorState(p.copy(), *[None if a is None else a.copy() for a in st], 8)
    ps = bnb8.ParamState(to_dev(p), None, *[to_dev(a) for a in st], 8)
    qd1 = to_dev(q1.copy())
    qd2 = None if q2 is None else to_dev(q2.copy())
    for k in range(1, 3):
        if k == 2:
            q1 = _moved_levels(q1, 42)
            qd1.copy_(to_dev(q1))
            if q2 is not None:
                q2 = _moved_levels(q2, 43)
                qd2.copy_(to_dev(q2))
        g = workloads.normal(n, 1e-2, 44 + k)
        ps.g = to_dev(g)
        hp = dict(HP_BASE[optim], step=k, weight_decay=1e-2)
        bnb8.step([ps], bnb8.HParams(optim=optim, **hp), qd1, qd2)
        oracle.step(oracle.HParams(optim=optim, **hp), ref, g, "f32", B, q1, q2)
        torch.cuda.synchronize()
        for name in ("p", "s1", "s2", "absmax1", "absmax2"):
            if getattr(ref, name) is not None:
                assert_same(f"{optim}/step{k}/{name}", to_host(getattr(ps, name)), getattr(ref, name))


# ---------------------------------------------------------------------------
# max_unorm per block (BNB8_UNORM_PER_BLOCK): the norms are formed inside the
# step; the multiplier matches the oracle's binary64 one to 1e-6, so p is
# compared at the max_unorm tolerance and codes / absmax bit for bit
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("optim", OPTIMS)
@pytest.mark.parametrize("mu", [0.05, 3.0])
def test_step_max_unorm_per_block(bnb8, qdev, optim, mu):
    run_case(bnb8, qdev, optim, "f32", [8, 32, 8], 256, [4000, 300, 256 * 9], steps=3,
             max_unorm=mu, wd=1e-2, seed=60, extra_hp=dict(unorm_per_block=True))


@pytest.mark.parametrize("B", [64, 2048])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_step_max_unorm_per_block_blocksizes(bnb8, qdev, B, dtype):
    run_case(bnb8, qdev, "adam", dtype, 8, B, [5 * B + 17, 3 * B], steps=2, max_unorm=0.5,
             seed=61, extra_hp=dict(unorm_per_block=True))


@pytest.mark.parametrize("optim", ["adam", "lion", "rmsprop", "ademamix"])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_skip_zeros_tensor_lists(bnb8, qdev, optim, dtype):
    """skip_zeros at B = 256 (the gradient-only ring) over a long list:
    whole-chunk and ragged tensors (launched apart), misaligned storage (the
    copies replaced by plain loads), and more tensors than one launch takes,
    so that the chunks a warp takes from its CTA's counter jump across
    tensors."""
    rng = np.random.default_rng(81)
    sizes = [int(x) for x in rng.integers(1, 2600, size=110)] + [512 * 7, 256 * 9 + 100, 1024 * 3]
    offsets = [1 if i % 17 == 5 else 0 for i in range(len(sizes))]
    run_case(bnb8, qdev, optim, dtype, 8, 256, sizes, steps=2, skip_zeros=True, zero_frac=0.4,
             wd=1e-2, seed=83, offsets=offsets)


@pytest.mark.parametrize("optim", ["adam", "lion", "rmsprop", "ademamix"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_step_max_unorm_per_tensor_skip_zeros(bnb8, qdev, optim, dtype):
    """Per-tensor max_unorm with skip_zeros: the pre-pass over a gradient
    with zero elements and all-zero blocks, the reduction, then the
    skip_zeros step (at B = 256 the gradient-only ring) applying each
    tensor's multiplier to its live blocks."""
    run_case(bnb8, qdev, optim, dtype, [8, 32, 8], 256, [6 * 512 + 100, 300, 256 * 9], steps=3,
             skip_zeros=True, zero_frac=0.3, wd=1e-2, max_unorm=0.05, seed=64)


@pytest.mark.parametrize("optim", ["adam", "momentum", "ademamix"])
def test_step_max_unorm_per_block_skip_zeros(bnb8, qdev, optim):
    run_case(bnb8, qdev, optim, "bf16", [8, 32], 256, [6 * 256 + 3, 700], steps=3,
             skip_zeros=True, zero_frac=0.2, wd=1e-2, max_unorm=0.5, seed=62,
             extra_hp=dict(unorm_per_block=True))


# ---------------------------------------------------------------------------
# tensor-wise quantization (blocksize 0): one absmax per state per tensor,
# the oracle taking each tensor as a single block
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("optim", OPTIMS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_step_tensorwise(bnb8, qdev, optim, dtype):
    run_case(bnb8, qdev, optim, dtype, 8, 0, [7 * 256 + 77, 300 * 256, 5], steps=3, wd=1e-2,
             seed=70)


@pytest.mark.parametrize("optim", ["adam", "momentum", "ademamix"])
def test_step_tensorwise_skip_zeros(bnb8, qdev, optim):
    run_case(bnb8, qdev, optim, "bf16", 8, 0, [20 * 256 + 3, 4000], steps=3, skip_zeros=True,
             zero_frac=0.3, wd=1e-2, seed=71)


def test_step_tensorwise_all_zero_gradient_untouched(bnb8, qdev):
    # skip_zeros with a gradient that is zero everywhere: codes, absmax and p
    # keep their bits (the oracle leaves the tensor's one block untouched)
    n = 5000
    st = random_state("adam", n, 8, n, 72, S, U)
    p = workloads.normal(n, 0.1, 73)
    ps = bnb8.ParamState(to_dev(p), to_dev(np.zeros(n, np.float32)), *[to_dev(a) for a in st], 8)
    bnb8.step([ps], bnb8.HParams(optim="adam", blocksize=0, skip_zeros=True, step=2), qdev[0],
              qdev[1])
    torch.cuda.synchronize()
    assert_same("p", to_host(ps.p), p)
    for got, want in zip((ps.s1, ps.s2, ps.absmax1, ps.absmax2), st):
        assert_same("state", to_host(got), want)


def test_step_tensorwise_mixed_bits_and_max_unorm(bnb8, qdev):
    run_case(bnb8, qdev, "adam", "f32", [8, 32, 8], 0, [4000, 300, 256 * 9], steps=3,
             max_unorm=0.05, wd=1e-2, seed=74)


def test_tensorwise_rejects_per_block_unorm(bnb8, qdev):
    ps = bnb8.ParamState(torch.zeros(512, device="cuda"), torch.zeros(512, device="cuda"),
                         *bnb8.zero_state(torch.zeros(512, device="cuda"), "adam", 8, 0), 8)
    with pytest.raises(bnb8.Bnb8Error, match="tensor-wise"):
        bnb8.step([ps], bnb8.HParams(optim="adam", blocksize=0, max_unorm=1.0,
                                     unorm_per_block=True), qdev[0], qdev[1])


def test_step_tensorwise_list_over_launch_capacity(bnb8, qdev):
    # more tensors than one launch carries: the absmax accumulators are
    # indexed by the caller's list position across launches
    rng = np.random.default_rng(75)
    sizes = [int(x) for x in rng.integers(1, 3000, 130)]
    bits = [8 if n >= 1024 else 32 for n in sizes]
    run_case(bnb8, qdev, "adam", "bf16", bits, 0, sizes, steps=2, seed=76)


@pytest.mark.parametrize("blocksize,extra", [(0, {}), (256, dict(max_unorm=0.5, unorm_per_block=True))])
def test_stepper_with_options(bnb8, qdev, blocksize, extra):
    # tensor-wise (workspace) and per-block max_unorm through a Stepper
    n = 256 * 40 + 9
    st = random_state("adam", n, 8, blocksize or n, 80, S, U)
    p = workloads.normal(n, 0.1, 81)
    g = to_dev(workloads.normal(n, 1e-2, 82))
    a = bnb8.ParamState(to_dev(p), g, *[to_dev(x) for x in st], 8)
    b = bnb8.ParamState(to_dev(p), g, *[to_dev(x) for x in st], 8)
    hp = dict(HP_BASE["adam"], weight_decay=1e-2, blocksize=blocksize, **extra)
    stepper = bnb8.Stepper([b], bnb8.HParams(optim="adam", step=1, **hp), qdev[0], qdev[1])
    for k in range(1, 4):
        bnb8.step([a], bnb8.HParams(optim="adam", step=k, **hp), qdev[0], qdev[1])
        stepper(k)
    torch.cuda.synchronize()
    for name in ("p", "s1", "s2", "absmax1", "absmax2"):
        assert_same(name, to_host(getattr(b, name)), to_host(getattr(a, name)))
