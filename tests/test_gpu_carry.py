"""The carried parameter norm (hparams flag BNB8_CARRY_PNORM): a step with
max_unorm per tensor leaves the per-block sums of the new p^2 in its
workspace, and the next step's pre-pass takes ||p|| from them instead of
reading p.  docs page "optim_overview.md", max_unorm: the test compares the
update norm with max_unorm times the parameter norm; the carried norm is the
same quantity, formed while the step writes p.

Each step is checked two ways: the multipliers the step left in its workspace
against the oracle's definition on the step's own input (1e-6 relative), and
p and the states against the oracle's step given that multiplier (bit for
bit).  The mechanism tests change p behind the library's back (the one thing
the flag's contract forbids) to show that the norm was carried, and that
every documented invalidation recomputes it."""
import numpy as np
import pytest

import oracle
import workloads
from parity_util import assert_same, map_pair, maps, random_state, to_dev, to_host

S, U = maps()
pytestmark = pytest.mark.gpu


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


def _setup(bnb8, optim, dtype, sizes, bits, B, seed):
    q1, q2 = map_pair(optim, S, U)
    params = []
    for i, (n, b) in enumerate(zip(sizes, bits)):
        p = oracle.to_storage(workloads.normal(n, 0.05, seed + 10 * i), dtype)
        st = random_state(optim, n, b, B, seed + 10 * i + 1, q1, q2)
        params.append(bnb8.ParamState(to_dev(p, dtype), None, *[to_dev(a) for a in st], b))
    qd1 = to_dev(q1)
    qd2 = None if q2 is None else to_dev(q2)
    return params, q1, q2, qd1, qd2


def _snapshot(params):
    return [oracle.TensorState(to_host(ps.p), to_host(ps.s1), to_host(ps.s2), to_host(ps.absmax1),
                               to_host(ps.absmax2), ps.state_bits) for ps in params]


def _scales(ws, nt):
    # workspace layout: [stamp, 256 bytes][one float32 multiplier per tensor]...
    import torch
    return to_host(ws[256:256 + 4 * nt].view(torch.float32)).copy()


def _grads(params, dtype, k, seed):
    host = []
    for i, ps in enumerate(params):
        g = oracle.to_storage(workloads.normal(ps.p.numel(), 1e-2, seed + 1000 * k + i), dtype)
        host.append(g)
        ps.g = to_dev(g, dtype)
    return host


CASES = [
    # optimizer, dtype, sizes, bits, block, weight decay: the ring kernel (B >= 256,
    # several warps per block at 2048), the generic 8-bit kernel (B 128, AdEMAMix),
    # 32-bit states, ragged tails, and tensors of more than one 512-block chunk
    ("adam", "f32", [4000, 300, 256 * 1100 + 5], [8, 32, 8], 256, 0.0),
    ("adam", "f32", [5000, 256 * 9 + 17], [8, 8], 256, 1e-2),
    ("adamw", "bf16", [256 * 700 + 3, 3000, 777], [8, 8, 32], 256, 1e-2),
    ("lion", "bf16", [2048 * 5 + 300, 4100], [8, 8], 2048, 1e-2),
    ("momentum", "f32", [3000, 128 * 40 + 1], [8, 8], 128, 0.0),
    ("ademamix", "f32", [4096 + 256, 1000], [8, 32], 256, 1e-2),
    ("rmsprop", "f16", [5000, 2600], [8, 8], 256, 0.0),
    # fp32 blocks of 512 and more: the two-pass shape with the first pass parked
    ("adam", "f32", [2048 * 3 + 5, 4096], [8, 8], 2048, 1e-2),
    ("adamw", "f32", [512 * 7 + 100, 1024, 300], [8, 8, 32], 512, 1e-2),
]


@pytest.mark.parametrize("optim,dtype,sizes,bits,B,wd", CASES,
                         ids=[f"{c[0]}-{c[1]}-B{c[4]}-wd{c[5]}" for c in CASES])
def test_carried_norm_steps_match_the_oracle(bnb8, optim, dtype, sizes, bits, B, wd):
    import torch
    params, q1, q2, qd1, qd2 = _setup(bnb8, optim, dtype, sizes, bits, B, 300)
    base = dict(lr=1e-3, beta1=0.9, beta2=0.999, alpha=2.0, weight_decay=wd, max_unorm=0.02)
    if optim in ("momentum", "rmsprop"):
        base.update(lr=1e-2, beta1=0.9)
    ws = torch.empty(bnb8.bnb8_workspace_size(params, bnb8.HParams(optim=optim, blocksize=B,
                                                                   **base)),
                     dtype=torch.uint8, device="cuda")
    clipped = 0
    for k in range(1, 5):
        g = _grads(params, dtype, k, 310)
        before = _snapshot(params)
        bnb8.step(params, bnb8.HParams(optim=optim, blocksize=B, step=k, carry_pnorm=True, **base),
                  qd1, qd2, workspace=ws)
        torch.cuda.synchronize()
        got = _scales(ws, len(params))
        ohp = oracle.HParams(optim=optim, step=k, **base)
        for i, (ps, ref) in enumerate(zip(params, before)):
            want, _, _ = oracle.unorm_scale(ohp, ref, g[i], dtype, B, q1, q2)
            tag = f"{optim}/{dtype}/step{k}/t{i}"
            assert abs(float(got[i]) - want) <= 1e-6 * want, (tag, float(got[i]), want)
            clipped += want < 1.0
            # given the library's multiplier, the step itself is the oracle's, bit for bit
            oracle.step(ohp, ref, g[i], dtype, B, q1, q2, clip=float(got[i]))
            assert_same(tag + " p", to_host(ps.p), ref.p)
            assert_same(tag + " s1", to_host(ps.s1), ref.s1)
            assert_same(tag + " s2", to_host(ps.s2), ref.s2)
            assert_same(tag + " absmax1", to_host(ps.absmax1), ref.absmax1)
            assert_same(tag + " absmax2", to_host(ps.absmax2), ref.absmax2)
    assert clipped >= len(params)           # the clip was active in this case


def _changed_norm_case(bnb8, optim="adam", wd=0.0):
    # Adam without weight decay: the pre-pass needs p for nothing but ||p||
    import torch
    sizes, bits, B = [6000, 256 * 30 + 7, 900], [8, 8, 32], 256
    params, q1, q2, qd1, qd2 = _setup(bnb8, optim, "f32", sizes, bits, B, 400)
    base = dict(lr=1e-3, weight_decay=wd, max_unorm=0.02)
    ws = torch.empty(bnb8.bnb8_workspace_size(params, bnb8.HParams(optim=optim, **base)),
                     dtype=torch.uint8, device="cuda")
    return params, q1, q2, qd1, qd2, base, ws


def _step_and_check(bnb8, params, q1, q2, qd1, qd2, base, ws, k, stale_p, optim="adam",
                    carry=True, seed=410):
    """One step; its multipliers must be the definition's with ||p|| taken
    from stale_p (the p the carried sums describe), or from the current p
    when stale_p is None."""
    import torch
    g = _grads(params, "f32", k, seed)
    now = _snapshot(params)
    bnb8.step(params, bnb8.HParams(optim=optim, step=k, carry_pnorm=carry, **base), qd1, qd2,
              workspace=ws)
    torch.cuda.synchronize()
    got = _scales(ws, len(params))
    ohp = oracle.HParams(optim=optim, step=k, **base)
    for i, ref in enumerate(now):
        if stale_p is not None:
            ref = oracle.TensorState(stale_p[i], ref.s1, ref.s2, ref.absmax1, ref.absmax2,
                                     ref.state_bits)
        want, _, _ = oracle.unorm_scale(ohp, ref, g[i], "f32", 256, q1, q2)
        assert abs(float(got[i]) - want) <= 1e-6 * want, (k, i, float(got[i]), want)
    return got


def _double_p(params):
    old = [to_host(ps.p).copy() for ps in params]
    for ps in params:
        ps.p.mul_(2.0)
    return old


def test_the_norm_is_carried_and_every_invalidation_recomputes_it(bnb8):
    params, q1, q2, qd1, qd2, base, ws = _changed_norm_case(bnb8)
    args = (bnb8, params, q1, q2, qd1, qd2, base, ws)
    _step_and_check(*args, 1, None)
    # p changed behind the library's back: step 2 still uses the carried ||p||
    # (of the p step 1 left), which shows that it read no p for the norm
    old = _double_p(params)
    got = _step_and_check(*args, 2, old)
    # the same step number again: its stamp is step 2's, not step 1's -> recomputed
    _double_p(params)
    _step_and_check(*args, 2, None)
    # a pre-pass of the stand-alone entry point on the same workspace clears the stamp
    _step_and_check(*args, 3, None)
    bnb8.bnb8_unorm(params, bnb8.HParams(optim="adam", step=4, **base), qd1, qd2, workspace=ws)
    _double_p(params)
    _step_and_check(*args, 4, None)
    # a step without the flag clears it too
    _step_and_check(*args, 5, None, carry=False)
    _double_p(params)
    _step_and_check(*args, 6, None)
    assert np.all(got < 1.0)


def test_another_list_on_the_same_workspace_recomputes_the_norm(bnb8):
    import torch
    params, q1, q2, qd1, qd2, base, ws = _changed_norm_case(bnb8)
    args = (bnb8, params, q1, q2, qd1, qd2, base, ws)
    _step_and_check(*args, 1, None)
    # a second list (a sub-list of the first one's tensors) steps on the same
    # workspace; its pre-pass writes the partials and its stamp replaces ours
    other = [bnb8.ParamState(torch.randn(5000, device="cuda") * 0.05, None,
                             *[to_dev(a) for a in random_state("adam", 5000, 8, 256, 430, q1, q2)],
                             8)]
    _grads(other, "f32", 1, 440)
    bnb8.step(other, bnb8.HParams(optim="adam", step=2, carry_pnorm=True, **base), qd1, qd2,
              workspace=ws)
    _double_p(params)
    _step_and_check(*args, 2, None)


def test_coupled_decay_still_reads_p_for_the_direction(bnb8):
    # Adam with weight decay: the direction needs p, so the pre-pass reads it;
    # only ||p|| is carried.  With p doubled, U follows the current p while
    # ||p|| is the carried one.
    params, q1, q2, qd1, qd2, base, ws = _changed_norm_case(bnb8, wd=0.5)
    args = (bnb8, params, q1, q2, qd1, qd2, base, ws)
    _step_and_check(*args, 1, None)
    old = _double_p(params)
    import torch
    g = _grads(params, "f32", 2, 410)
    now = _snapshot(params)
    bnb8.step(params, bnb8.HParams(optim="adam", step=2, carry_pnorm=True, **base), qd1, qd2,
              workspace=ws)
    torch.cuda.synchronize()
    got = _scales(ws, len(params))
    ohp = oracle.HParams(optim="adam", step=2, **base)
    for i, ref in enumerate(now):
        _, unorm, _ = oracle.unorm_scale(ohp, ref, g[i], "f32", 256, q1, q2)
        pnorm = np.sqrt(oracle.param_sumsq(old[i], "f32"))
        limit = base["max_unorm"] * pnorm
        want = limit / unorm if unorm > limit else 1.0
        assert abs(float(got[i]) - want) <= 1e-6 * want, (i, float(got[i]), want)
