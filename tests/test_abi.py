"""The C-ABI library on the host (no GPU needed): it loads, exports every
symbol include/bnb8.h declares, creates the map bit-identically to the oracle,
and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest

import bit_block_wise_gb300 as bnb8
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from bit_block_wise_gb300 import build
    build.build()
    return bnb8.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "bnb8.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bnb8_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) == 16
    assert sorted(bnb8.EXPORTS) == names
    for name in names:
        assert hasattr(L, name), name


def test_struct_layouts_match_header():
    assert ctypes.sizeof(bnb8.Bnb8Tensor) == 64
    assert ctypes.sizeof(bnb8.Bnb8Hparams) == 80
    assert bnb8.Bnb8Hparams.step.offset == 56


def test_version(L):
    assert bnb8.bnb8_version() >= 100


@pytest.mark.parametrize("signed", [True, False])
def test_create_qmap_matches_oracle(L, signed):
    q = bnb8.bnb8_create_qmap(signed).numpy()
    np.testing.assert_array_equal(q, oracle.create_qmap(signed))


def test_create_qmap_null(L):
    assert L.bnb8_create_qmap(1, None) == bnb8.BNB8_EINVAL
    assert b"NULL" in L.bnb8_last_error()


@pytest.mark.parametrize("signed", [True, False])
def test_qmap_code_matches_oracle_rule(L, signed):
    q = oracle.create_qmap(signed)
    mid = oracle.midpoints(q)
    rng = np.random.default_rng(5)
    xs = np.concatenate([q, mid, np.nextafter(mid, np.float32(2)), np.nextafter(mid, np.float32(-2)),
                         rng.uniform(-1.0, 1.0, 200).astype(np.float32), [0.0, -0.0, 2.0, -2.0]])
    for x in xs.astype(np.float32):
        assert bnb8.bnb8_qmap_code(q, float(x)) == oracle.code(mid, float(x)), x


def test_zero_state_codes_come_from_the_map(L):
    import torch
    p = torch.zeros(1000)
    s1, s2, a1, a2 = bnb8.zero_state(p, "adam", 8, 256)
    S, U = oracle.create_qmap(True), oracle.create_qmap(False)
    assert int(s1[0]) == int(np.count_nonzero(oracle.midpoints(S) < 0))
    assert int(s2[0]) == int(np.count_nonzero(oracle.midpoints(U) < 0))
    # a caller's map whose 0.0 sits at index 40: its zero state holds code 40
    custom = np.concatenate([np.linspace(-1.0, -0.01, 40), [0.0],
                             np.linspace(0.005, 1.0, 215)]).astype(np.float32)
    assert np.all(np.diff(custom) > 0) and custom.size == 256
    s1, s2, _, _ = bnb8.zero_state(p, "adam", 8, 256, qmap1=torch.from_numpy(custom))
    assert torch.all(s1 == 40) and torch.all(s2 == int(s2[0])) and int(s2[0]) == 0
    s1, _, _, _ = bnb8.zero_state(p, "rmsprop", 8, 256, qmap1=torch.from_numpy(custom))
    assert torch.all(s1 == 40)


def test_qmap_code_rejects_bad_maps(L):
    q = oracle.create_qmap(True)
    out = ctypes.c_uint8()
    assert L.bnb8_qmap_code(None, 0.0, ctypes.byref(out)) == bnb8.BNB8_EINVAL
    assert L.bnb8_qmap_code(q.ctypes.data, float("nan"), ctypes.byref(out)) == bnb8.BNB8_EINVAL
    bad = q.copy()
    bad[100] = bad[99]
    assert L.bnb8_qmap_code(bad.ctypes.data, 0.0, ctypes.byref(out)) == bnb8.BNB8_EINVAL
    assert b"ascending" in L.bnb8_last_error()


def _hp(**kw):
    base = dict(optim=bnb8.BNB8_ADAM, dtype=bnb8.BNB8_F32, blocksize=256, skip_zeros=0, lr=1e-3,
                beta1=0.9, beta2=0.999, beta3=0.9999, alpha=0.0, eps=1e-8, weight_decay=0.0,
                gnorm_scale=1.0, max_unorm=0.0, flags=0, step=1, t_alpha=0, t_beta3=0)
    base.update(kw)
    return bnb8.Bnb8Hparams(**base)


FAKE = 0x7f0000000000  # never dereferenced: every case below fails validation first


def _tensor(**kw):
    base = dict(p=FAKE, g=FAKE + 4096, s1=FAKE + 8192, s2=FAKE + 12288, absmax1=FAKE + 16384,
                absmax2=FAKE + 20480, n=1000, state_bits=8, reserved=0)
    base.update(kw)
    return bnb8.Bnb8Tensor(**base)


def _call2(L, tensors, hp, q1=FAKE, q2=FAKE, ws=None, wsb=0):
    arr = (bnb8.Bnb8Tensor * max(1, len(tensors)))(*tensors)
    return L.bnb8_step_2state(arr, len(tensors), ctypes.byref(hp), q1, q2, ws, wsb, None)


@pytest.mark.parametrize("kw,frag", [
    (dict(blocksize=100), b"blocksize"),
    (dict(blocksize=32), b"blocksize"),
    (dict(blocksize=8192), b"blocksize"),
    (dict(dtype=7), b"dtype"),
    (dict(optim=bnb8.BNB8_LION), b"optimizer"),
    (dict(step=0), b"step"),
    (dict(flags=4), b"flags"),
    (dict(max_unorm=-1.0), b"max_unorm"),
    (dict(max_unorm=float("nan")), b"max_unorm"),
    (dict(t_alpha=-1), b"t_alpha"),
])
def test_bad_hparams_rejected(L, kw, frag):
    assert _call2(L, [_tensor()], _hp(**kw)) == bnb8.BNB8_EINVAL
    assert frag in L.bnb8_last_error()


@pytest.mark.parametrize("kw,frag", [
    (dict(n=-1), b"n < 0"),
    (dict(p=0), b"NULL"),
    (dict(g=0), b"NULL"),
    (dict(s1=0), b"NULL"),
    (dict(s2=0), b"s2"),
    (dict(absmax1=0), b"absmax"),
    (dict(state_bits=16), b"state_bits"),
    (dict(p=FAKE + 2), b"aligned"),
    (dict(reserved=3), b"reserved"),
])
def test_bad_tensor_rejected(L, kw, frag):
    assert _call2(L, [_tensor(), _tensor(**kw)], _hp()) == bnb8.BNB8_EINVAL
    msg = L.bnb8_last_error()
    assert frag in msg and b"tensor 1" in msg


def test_missing_qmap_rejected(L):
    assert _call2(L, [_tensor()], _hp(), q1=None) == bnb8.BNB8_EINVAL
    assert b"qmap" in L.bnb8_last_error()


def test_entry_point_optimizer_mismatch(L):
    arr = (bnb8.Bnb8Tensor * 1)(_tensor())
    hp = _hp(optim=bnb8.BNB8_ADAM)
    assert L.bnb8_step_1state(arr, 1, ctypes.byref(hp), FAKE, None, 0, None) == bnb8.BNB8_EINVAL
    assert L.bnb8_step_ademamix(arr, 1, ctypes.byref(hp), FAKE, FAKE, None, 0,
                                None) == bnb8.BNB8_EINVAL


def test_workspace_size_and_check(L):
    ts = [_tensor(n=1000), _tensor(n=256 * 3), _tensor(n=0), _tensor(n=5, state_bits=32)]
    arr = (bnb8.Bnb8Tensor * 4)(*ts)
    assert L.bnb8_workspace_size(arr, 4, ctypes.byref(_hp())) == 0       # max_unorm off
    hp = _hp(max_unorm=1.0)
    need = L.bnb8_workspace_size(arr, 4, ctypes.byref(hp))
    blocks = 4 + 3 + 0 + 1
    # the carried norm's stamp, the multipliers, one float2 partial per block,
    # the reduction's tickets (one word for each of up to 96 tensors a launch)
    assert need == 256 + 256 + ((blocks * 8 + 255) // 256) * 256 + 512
    assert _call2(L, ts, hp, ws=None, wsb=0) == bnb8.BNB8_EWORKSPACE
    assert _call2(L, ts, hp, ws=FAKE, wsb=need - 1) == bnb8.BNB8_EWORKSPACE
    assert _call2(L, ts, hp, ws=FAKE + 8, wsb=need) == bnb8.BNB8_EWORKSPACE
    assert b"workspace" in L.bnb8_last_error()


def test_per_block_unorm_needs_no_workspace(L):
    ts = [_tensor(n=1000), _tensor(n=5, state_bits=32)]
    arr = (bnb8.Bnb8Tensor * 2)(*ts)
    hp = _hp(max_unorm=1.0, flags=bnb8.BNB8_UNORM_PER_BLOCK)
    assert L.bnb8_workspace_size(arr, 2, ctypes.byref(hp)) == 0
    # the per-tensor pre-pass entry points refuse it
    assert L.bnb8_unorm(arr, 2, ctypes.byref(hp), FAKE, FAKE, FAKE, None, 0, None) == bnb8.BNB8_EINVAL
    assert b"per-tensor" in L.bnb8_last_error()
    assert L.bnb8_unorm_static(arr, 2, ctypes.byref(hp), FAKE, FAKE, FAKE, None) == bnb8.BNB8_EINVAL


def test_quantize_args_rejected(L):
    assert L.bnb8_quantize_blockwise(FAKE, 0, 10, FAKE, 96, FAKE, FAKE, None) == bnb8.BNB8_EINVAL
    assert L.bnb8_quantize_blockwise(FAKE, 3, 10, FAKE, 256, FAKE, FAKE, None) == bnb8.BNB8_EINVAL
    assert L.bnb8_quantize_blockwise(None, 0, 10, FAKE, 256, FAKE, FAKE, None) == bnb8.BNB8_EINVAL
    assert L.bnb8_quantize_blockwise(FAKE, 0, -1, FAKE, 256, FAKE, FAKE, None) == bnb8.BNB8_EINVAL
    assert L.bnb8_quantize_blockwise(None, 0, 0, None, 256, None, None, None) == bnb8.BNB8_OK
    assert L.bnb8_dequantize_blockwise(FAKE, FAKE, FAKE, 256, 10, FAKE + 1, 0,
                                       None) == bnb8.BNB8_EINVAL


def test_empty_lists_are_noops(L):
    hp = _hp()
    assert L.bnb8_step_2state(None, 0, ctypes.byref(hp), None, None, None, 0, None) == bnb8.BNB8_OK
    assert _call2(L, [_tensor(n=0)], hp, q1=None, q2=None) == bnb8.BNB8_OK


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(bnb8, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(bnb8, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        bnb8.lib()


def test_launch_block_limit(L):
    # the 8-bit kernels index one launch's blocks with 32-bit integers: a list
    # beyond 2^31 - 1 blocks is refused before any device work
    t = _tensor(n=(1 << 31) * 256 + 1)
    assert _call2(L, [t], _hp()) == bnb8.BNB8_EUNSUPPORTED
    assert b"blocks in one launch" in L.bnb8_last_error()


def test_paged_args_rejected_before_the_device(L):
    out = ctypes.c_void_p(1234)
    assert L.bnb8_paged_alloc(0, ctypes.byref(out)) == bnb8.BNB8_EINVAL
    assert out.value is None  # cleared on failure
    assert L.bnb8_paged_alloc(16, None) == bnb8.BNB8_EINVAL
    assert L.bnb8_paged_prefetch(None, 16, 0, None) == bnb8.BNB8_EINVAL
    assert L.bnb8_paged_prefetch(ctypes.c_void_p(4096), 16, -2, None) == bnb8.BNB8_EINVAL
    assert b"BNB8_PAGED_HOST" in L.bnb8_last_error()
    assert L.bnb8_paged_prefetch(None, 0, 0, None) == bnb8.BNB8_OK  # nothing to move
    assert L.bnb8_paged_free(None) == bnb8.BNB8_OK
