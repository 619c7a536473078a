"""Oracle for the 8-bit block-wise dynamic-quantized optimizer step.

TEST INFRASTRUCTURE ONLY.  This package wraps ``bnb8_oracle.c`` -- a plain,
single-threaded C statement of the method -- with ctypes and numpy.  Only the
test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it; the GPU library never does, and the two share no
code.

Arrays are numpy: float32 tensors as ``np.float32``; bfloat16 and float16
tensors as their raw 16-bit patterns in ``np.uint16``; codes as ``np.uint8``;
absmax as ``np.float32``.  All calls mutate their state arguments in place,
like the optimizer does.
"""
from __future__ import annotations

import contextlib
import ctypes
import dataclasses
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bnb8_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_bnb8.so")

# Compiler flags: every binary32 operation rounded once, in source order.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

DTYPES = {"f32": 0, "bf16": 1, "f16": 2}
OPTIMS = {
    "adam": 0,
    "adamw": 1,
    "momentum": 2,
    "rmsprop": 3,
    "adagrad": 4,
    "lion": 5,
    "ademamix": 6,
}
NSTATES = {"adam": 2, "adamw": 2, "momentum": 1, "rmsprop": 1, "adagrad": 1, "lion": 1,
           "ademamix": 3}


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (idempotent)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _HParams(ctypes.Structure):
    _fields_ = [
        ("optim", ctypes.c_int),
        ("lr", ctypes.c_float),
        ("beta1", ctypes.c_float),
        ("beta2", ctypes.c_float),
        ("beta3", ctypes.c_float),
        ("alpha", ctypes.c_float),
        ("eps", ctypes.c_float),
        ("weight_decay", ctypes.c_float),
        ("gnorm_scale", ctypes.c_float),
        ("max_unorm", ctypes.c_float),
        ("step", ctypes.c_int64),
        ("t_alpha", ctypes.c_int64),
        ("t_beta3", ctypes.c_int64),
        ("skip_zeros", ctypes.c_int),
        ("unorm_per_block", ctypes.c_int),
    ]


class _Scalars(ctypes.Structure):
    _fields_ = [
        ("b1", ctypes.c_float),
        ("b2", ctypes.c_float),
        ("b3t", ctypes.c_float),
        ("omb1", ctypes.c_float),
        ("omb2", ctypes.c_float),
        ("omb3t", ctypes.c_float),
        ("step_size", ctypes.c_float),
        ("eps_hat", ctypes.c_float),
        ("inv_bc1", ctypes.c_float),
        ("alpha_t", ctypes.c_float),
        ("decay", ctypes.c_float),
        ("unorm_c", ctypes.c_double),
    ]


_lib = None


def _configure(L):
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    L.oracle_create_qmap.argtypes = [ctypes.c_int, vp]
    L.oracle_midpoints.argtypes = [vp, vp]
    L.oracle_code.argtypes = [vp, ctypes.c_float]
    L.oracle_code.restype = ctypes.c_int
    L.oracle_quantize_blockwise.argtypes = [vp, ctypes.c_int, i64, vp, i64, vp, vp]
    L.oracle_dequantize_blockwise.argtypes = [vp, vp, vp, i64, i64, vp, ctypes.c_int]
    L.oracle_scalars.argtypes = [ctypes.POINTER(_HParams), ctypes.POINTER(_Scalars)]
    L.oracle_unorm_scale.argtypes = [ctypes.POINTER(_HParams), vp, vp, vp, vp, vp, vp, i64,
                                     ctypes.c_int, ctypes.c_int, i64, vp, vp,
                                     ctypes.POINTER(ctypes.c_double),
                                     ctypes.POINTER(ctypes.c_double)]
    L.oracle_unorm_scale.restype = ctypes.c_float
    L.oracle_param_sumsq.argtypes = [vp, ctypes.c_int, i64]
    L.oracle_param_sumsq.restype = ctypes.c_double
    L.oracle_step.argtypes = [ctypes.POINTER(_HParams), vp, vp, vp, vp, vp, vp, i64,
                              ctypes.c_int, ctypes.c_int, i64, vp, vp]
    L.oracle_step.restype = ctypes.c_float
    L.oracle_step_clipped.argtypes = L.oracle_step.argtypes + [ctypes.c_float]
    L.oracle_step_clipped.restype = ctypes.c_float
    L.oracle_convert.argtypes = [vp, i64, vp, ctypes.c_int]
    L.oracle_widen.argtypes = [vp, ctypes.c_int, i64, vp]
    return L


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = _configure(ctypes.CDLL(_LIB_PATH))
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Run the oracle API against another build of the C source (the test
    suite plants mistakes in copies of it to show that the pins catch them)."""
    global _lib
    saved = _lib
    _lib = _configure(ctypes.CDLL(path))
    try:
        yield _lib
    finally:
        _lib = saved


def compile_variant(source_text: str, out_path: str) -> str:
    """Compile C source text with the oracle's flags into out_path."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.check_call(["gcc", *CFLAGS, "-o", out_path, src, "-lm"])
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


@dataclasses.dataclass
class HParams:
    """Hyperparameters of one update.

    Defaults follow the bitsandbytes docs page "optim_overview.md"
    (Optimizer2State: lr 1e-3, betas (0.9, 0.999), eps 1e-8, weight_decay 0,
    max_unorm 0.0, skip_zeros False, alpha 0.0, t_alpha/t_beta3 None).
    ``beta3`` is AdEMAMix's third beta; ``gnorm_scale`` multiplies the raw
    gradient.  ``step`` is the 1-based number of the update being taken.
    ``unorm_per_block`` takes max_unorm per block of ``blocksize`` elements
    (one multiplier per block) instead of per tensor.
    """
    optim: str = "adam"
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    beta3: float = 0.9999
    alpha: float = 0.0
    eps: float = 1e-8
    weight_decay: float = 0.0
    gnorm_scale: float = 1.0
    max_unorm: float = 0.0
    step: int = 1
    t_alpha: int = 0
    t_beta3: int = 0
    skip_zeros: bool = False
    unorm_per_block: bool = False

    def c(self) -> _HParams:
        return _HParams(OPTIMS[self.optim], self.lr, self.beta1, self.beta2, self.beta3,
                        self.alpha, self.eps, self.weight_decay, self.gnorm_scale,
                        self.max_unorm, int(self.step), int(self.t_alpha), int(self.t_beta3),
                        int(bool(self.skip_zeros)), int(bool(self.unorm_per_block)))


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be contiguous"
    return a.ctypes.data


def _storage_dtype(dtype: str):
    return np.float32 if dtype == "f32" else np.uint16


# ---- dtype conversion --------------------------------------------------------
def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to ``dtype`` storage (nearest even)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=_storage_dtype(dtype))
    lib().oracle_convert(_ptr(x), x.size, _ptr(out), DTYPES[dtype])
    return out


def to_f32(x: np.ndarray, dtype: str) -> np.ndarray:
    """Widen ``dtype`` storage to float32 (exact)."""
    x = np.ascontiguousarray(x)
    out = np.empty(x.shape, dtype=np.float32)
    lib().oracle_widen(_ptr(x), DTYPES[dtype], x.size, _ptr(out))
    return out


# ---- map, search, block-wise quantization ----------------------------------
def create_qmap(signed: bool) -> np.ndarray:
    out = np.empty(256, dtype=np.float32)
    lib().oracle_create_qmap(int(bool(signed)), _ptr(out))
    return out


def midpoints(q: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.float32)
    out = np.empty(255, dtype=np.float32)
    lib().oracle_midpoints(_ptr(q), _ptr(out))
    return out


def code(mid: np.ndarray, xn: float) -> int:
    mid = np.ascontiguousarray(mid, dtype=np.float32)
    return int(lib().oracle_code(_ptr(mid), float(xn)))


def quantize_blockwise(x: np.ndarray, dtype: str, q: np.ndarray, blocksize: int):
    x = np.ascontiguousarray(x)
    n = x.size
    nb = (n + blocksize - 1) // blocksize
    codes = np.empty(n, dtype=np.uint8)
    absmax = np.empty(nb, dtype=np.float32)
    q = np.ascontiguousarray(q, dtype=np.float32)
    lib().oracle_quantize_blockwise(_ptr(x), DTYPES[dtype], n, _ptr(q), blocksize, _ptr(codes),
                                    _ptr(absmax))
    return codes, absmax


def dequantize_blockwise(codes: np.ndarray, absmax: np.ndarray, q: np.ndarray, blocksize: int,
                         dtype: str = "f32") -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    absmax = np.ascontiguousarray(absmax, dtype=np.float32)
    q = np.ascontiguousarray(q, dtype=np.float32)
    out = np.empty(codes.size, dtype=_storage_dtype(dtype))
    lib().oracle_dequantize_blockwise(_ptr(codes), _ptr(absmax), _ptr(q), blocksize, codes.size,
                                      _ptr(out), DTYPES[dtype])
    return out


# ---- optimizer step ----------------------------------------------------------
def scalars(hp: HParams) -> dict:
    hc = hp.c()
    sc = _Scalars()
    lib().oracle_scalars(ctypes.byref(hc), ctypes.byref(sc))
    return {name: getattr(sc, name) for name, _ in _Scalars._fields_}


@dataclasses.dataclass
class TensorState:
    """One parameter tensor and its optimizer state.

    8-bit: ``s1``/``s2`` are uint8 codes and ``absmax1``/``absmax2`` float32
    per block.  32-bit: ``s1``/``s2`` are float32 and the absmax arrays None.
    AdEMAMix keeps m1 and m2 stacked in ``s1`` ([2, n]) and ``absmax1``
    ([2, nblocks]); nu is ``s2``.  Unused slots are None.
    """
    p: np.ndarray
    s1: np.ndarray
    s2: np.ndarray | None
    absmax1: np.ndarray | None
    absmax2: np.ndarray | None
    state_bits: int

    def copy(self) -> "TensorState":
        cp = lambda a: None if a is None else a.copy()
        return TensorState(self.p.copy(), cp(self.s1), cp(self.s2), cp(self.absmax1),
                           cp(self.absmax2), self.state_bits)


def zero_state(optim: str, n: int, state_bits: int, blocksize: int, q1=None, q2=None):
    """Optimizer state equal to all-zero binary32 states (the code of 0.0 and
    absmax 0 for 8-bit states)."""
    k = NSTATES[optim]
    if state_bits == 32:
        s1 = np.zeros(n * (2 if optim == "ademamix" else 1), dtype=np.float32)
        s2 = np.zeros(n, dtype=np.float32) if k >= 2 else None
        return s1, s2, None, None
    nb = (n + blocksize - 1) // blocksize
    zc1 = int(np.count_nonzero(midpoints(q1) < 0.0))
    s1 = np.full(n * (2 if optim == "ademamix" else 1), zc1, dtype=np.uint8)
    a1 = np.zeros(nb * (2 if optim == "ademamix" else 1), dtype=np.float32)
    s2 = a2 = None
    if k >= 2:
        zc2 = int(np.count_nonzero(midpoints(q2) < 0.0))
        s2 = np.full(n, zc2, dtype=np.uint8)
        a2 = np.zeros(nb, dtype=np.float32)
    return s1, s2, a1, a2


def unorm_scale(hp: HParams, t: TensorState, g: np.ndarray, dtype: str, blocksize: int,
                q1=None, q2=None):
    """Step multiplier from max_unorm, and the two norms (update, parameter)."""
    hc = hp.c()
    U = ctypes.c_double()
    P = ctypes.c_double()
    s = lib().oracle_unorm_scale(ctypes.byref(hc), _ptr(t.p), _ptr(g), _ptr(t.s1), _ptr(t.s2),
                                 _ptr(t.absmax1), _ptr(t.absmax2), t.p.size, t.state_bits,
                                 DTYPES[dtype], blocksize, _ptr(q1), _ptr(q2), ctypes.byref(U),
                                 ctypes.byref(P))
    return float(s), U.value, P.value


def param_sumsq(p: np.ndarray, dtype: str) -> float:
    """Sum of p^2 in binary64, in element order (p stored as ``dtype``): the
    squared P of the max_unorm test, for the next step when p is the
    parameter a step has just left."""
    p = np.ascontiguousarray(p)
    return float(lib().oracle_param_sumsq(_ptr(p), DTYPES[dtype], p.size))


def step(hp: HParams, t: TensorState, g: np.ndarray, dtype: str, blocksize: int, q1=None,
         q2=None, clip: float | None = None) -> float:
    """One optimizer update of tensor ``t`` in place; returns the clip multiplier.
    ``clip`` (>= 0) supplies the max_unorm multiplier of the whole tensor when
    ``t`` holds only some of its blocks."""
    hc = hp.c()
    if t.state_bits == 8:
        assert q1 is not None and (NSTATES[hp.optim] == 1 or q2 is not None)
        q1 = np.ascontiguousarray(q1, dtype=np.float32)
        q2 = None if q2 is None else np.ascontiguousarray(q2, dtype=np.float32)
    return float(lib().oracle_step_clipped(
        ctypes.byref(hc), _ptr(t.p), _ptr(g), _ptr(t.s1), _ptr(t.s2), _ptr(t.absmax1),
        _ptr(t.absmax2), t.p.size, t.state_bits, DTYPES[dtype], blocksize, _ptr(q1), _ptr(q2),
        -1.0 if clip is None else float(clip)))
