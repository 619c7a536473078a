"""Python binding of the GB300 8-bit block-wise optimizer library (libbnb8.so).

Argument marshalling only: every function here packs torch tensors (device
memory owned by the caller) into the C structures of ``include/bnb8.h`` and
calls the entry point of the same name.  All computation runs in the CUDA
kernels of the library; there is no CPU path.  If the library has not been
built, or no CUDA device is present, calls raise ``RuntimeError``.

The optimizer method is the 8-bit block-wise dynamic-quantized step of
"8-bit Optimizers via Block-wise Quantization" (Dettmers et al.) with the
optimizer set and parameters of the bitsandbytes docs page "optim_overview.md".
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbnb8.so")

BNB8_OK, BNB8_EINVAL, BNB8_EUNSUPPORTED, BNB8_ECUDA, BNB8_EWORKSPACE = 0, 1, 2, 3, 4
BNB8_F32, BNB8_BF16, BNB8_F16 = 0, 1, 2
BNB8_ADAM, BNB8_ADAMW, BNB8_MOMENTUM, BNB8_RMSPROP, BNB8_ADAGRAD, BNB8_LION, BNB8_ADEMAMIX = range(7)
BNB8_UNORM_PER_BLOCK = 1
BNB8_CARRY_PNORM = 2
BNB8_TEST_STALL_WAIT = 0x100
BNB8_STATUS_WAIT_TIMEOUT = 1
BNB8_PAGED_HOST = -1

OPTIMS = {"adam": BNB8_ADAM, "adamw": BNB8_ADAMW, "momentum": BNB8_MOMENTUM,
          "rmsprop": BNB8_RMSPROP, "adagrad": BNB8_ADAGRAD, "lion": BNB8_LION,
          "ademamix": BNB8_ADEMAMIX}
NSTATES = {"adam": 2, "adamw": 2, "momentum": 1, "rmsprop": 1, "adagrad": 1, "lion": 1,
           "ademamix": 3}
# bitsandbytes docs page "optim_overview.md": tensors below min_8bit_size
# elements keep 32-bit state.
MIN_8BIT_SIZE = 4096

# every symbol include/bnb8.h declares
EXPORTS = ("bnb8_last_error", "bnb8_version", "bnb8_create_qmap", "bnb8_qmap_code",
           "bnb8_quantize_blockwise",
           "bnb8_dequantize_blockwise", "bnb8_workspace_size", "bnb8_step_2state",
           "bnb8_step_1state", "bnb8_step_ademamix", "bnb8_unorm", "bnb8_unorm_static",
           "bnb8_paged_alloc", "bnb8_paged_prefetch", "bnb8_paged_free", "bnb8_device_status")


class Bnb8Tensor(ctypes.Structure):
    _fields_ = [("p", ctypes.c_void_p), ("g", ctypes.c_void_p), ("s1", ctypes.c_void_p),
                ("s2", ctypes.c_void_p), ("absmax1", ctypes.c_void_p),
                ("absmax2", ctypes.c_void_p), ("n", ctypes.c_int64),
                ("state_bits", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class Bnb8Hparams(ctypes.Structure):
    _fields_ = [("optim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("blocksize", ctypes.c_int32), ("skip_zeros", ctypes.c_int32),
                ("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("beta3", ctypes.c_float), ("alpha", ctypes.c_float), ("eps", ctypes.c_float),
                ("weight_decay", ctypes.c_float), ("gnorm_scale", ctypes.c_float),
                ("max_unorm", ctypes.c_float), ("flags", ctypes.c_int32),
                ("step", ctypes.c_int64), ("t_alpha", ctypes.c_int64),
                ("t_beta3", ctypes.c_int64)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C library (raises RuntimeError if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.bnb8_last_error.restype = ctypes.c_char_p
        L.bnb8_last_error.argtypes = []
        L.bnb8_version.restype = i32
        L.bnb8_create_qmap.argtypes = [i32, vp]
        L.bnb8_qmap_code.argtypes = [vp, ctypes.c_float, ctypes.POINTER(ctypes.c_uint8)]
        L.bnb8_quantize_blockwise.argtypes = [vp, i32, i64, vp, i32, vp, vp, vp]
        L.bnb8_dequantize_blockwise.argtypes = [vp, vp, vp, i32, i64, vp, i32, vp]
        L.bnb8_workspace_size.argtypes = [ctypes.POINTER(Bnb8Tensor), i32,
                                          ctypes.POINTER(Bnb8Hparams)]
        L.bnb8_workspace_size.restype = ctypes.c_size_t
        for name in ("bnb8_step_2state", "bnb8_step_ademamix"):
            getattr(L, name).argtypes = [ctypes.POINTER(Bnb8Tensor), i32,
                                         ctypes.POINTER(Bnb8Hparams), vp, vp, vp,
                                         ctypes.c_size_t, vp]
        L.bnb8_step_1state.argtypes = [ctypes.POINTER(Bnb8Tensor), i32,
                                       ctypes.POINTER(Bnb8Hparams), vp, vp, ctypes.c_size_t, vp]
        L.bnb8_unorm.argtypes = [ctypes.POINTER(Bnb8Tensor), i32, ctypes.POINTER(Bnb8Hparams),
                                 vp, vp, vp, vp, ctypes.c_size_t, vp]
        L.bnb8_unorm_static.argtypes = [ctypes.POINTER(Bnb8Tensor), i32,
                                        ctypes.POINTER(Bnb8Hparams), vp, vp, vp, vp]
        L.bnb8_paged_alloc.argtypes = [ctypes.c_size_t, ctypes.POINTER(ctypes.c_void_p)]
        L.bnb8_paged_prefetch.argtypes = [vp, ctypes.c_size_t, i32, vp]
        L.bnb8_paged_free.argtypes = [vp]
        L.bnb8_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
        for name in EXPORTS:
            if name not in ("bnb8_last_error", "bnb8_version", "bnb8_workspace_size"):
                getattr(L, name).restype = i32
        _lib = L
    return _lib


class Bnb8Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"bnb8 status {status}: {message}")
        self.status = status


def _check(status: int) -> None:
    if status != BNB8_OK:
        raise Bnb8Error(status, lib().bnb8_last_error().decode())


def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dtype_code(t) -> int:
    torch = _torch()
    return {torch.float32: BNB8_F32, torch.bfloat16: BNB8_BF16, torch.float16: BNB8_F16}[t.dtype]


def _stream(stream) -> Optional[int]:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# ---- hyperparameters -----------------------------------------------------------

@dataclasses.dataclass
class HParams:
    """Hyperparameters of one update (defaults: docs page "optim_overview.md",
    Optimizer2State).  ``step`` is the 1-based number of this update."""
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
    blocksize: int = 256
    unorm_per_block: bool = False  # max_unorm per block (BNB8_UNORM_PER_BLOCK)
    carry_pnorm: bool = False      # carry ||p|| to the next step (BNB8_CARRY_PNORM)
    extra_flags: int = 0           # other hparams.flags bits (BNB8_TEST_STALL_WAIT)

    def c(self, dtype_code: int) -> Bnb8Hparams:
        flags = ((BNB8_UNORM_PER_BLOCK if self.unorm_per_block else 0) |
                 (BNB8_CARRY_PNORM if self.carry_pnorm else 0) | int(self.extra_flags))
        return Bnb8Hparams(OPTIMS[self.optim], dtype_code, self.blocksize, int(bool(self.skip_zeros)),
                           self.lr, self.beta1, self.beta2, self.beta3, self.alpha, self.eps,
                           self.weight_decay, self.gnorm_scale, self.max_unorm, flags,
                           int(self.step), int(self.t_alpha), int(self.t_beta3))


@dataclasses.dataclass
class ParamState:
    """A parameter, its gradient and its optimizer state (torch tensors on the
    device).  8-bit: s1/s2 uint8 codes with float32 absmax1/absmax2; 32-bit:
    s1/s2 float32 and absmax None.  AdEMAMix: s1 = [2, n] (m1, m2),
    absmax1 = [2, nblocks], s2 = nu."""
    p: object
    g: object
    s1: object
    s2: object = None
    absmax1: object = None
    absmax2: object = None
    state_bits: int = 8

    def c(self) -> Bnb8Tensor:
        return Bnb8Tensor(_ptr(self.p), _ptr(self.g), _ptr(self.s1), _ptr(self.s2),
                          _ptr(self.absmax1), _ptr(self.absmax2), self.p.numel(),
                          self.state_bits, 0)


def _tensor_array(params: Sequence[ParamState]):
    arr = (Bnb8Tensor * max(1, len(params)))()
    for i, ps in enumerate(params):
        arr[i] = ps.c()
    return arr


# ---- entry points (same names as include/bnb8.h) -----------------------------

def bnb8_version() -> int:
    return int(lib().bnb8_version())


def bnb8_device_status(clear: bool = False) -> int:
    """The library's device status word of the current device (bits
    BNB8_STATUS_*), read after the device finishes its work; clear zeroes it."""
    out = ctypes.c_uint32()
    _check(lib().bnb8_device_status(ctypes.byref(out), int(bool(clear))))
    return int(out.value)


def bnb8_create_qmap(is_signed: bool):
    """The 256-level dynamic map as a float32 CPU tensor."""
    torch = _torch()
    out = torch.empty(256, dtype=torch.float32)
    _check(lib().bnb8_create_qmap(int(bool(is_signed)), out.data_ptr()))
    return out


def bnb8_qmap_code(qmap, x: float) -> int:
    """The code of the normalised value x under a map (any 256-element
    float32 tensor or array; copied to the host)."""
    torch = _torch()
    q = torch.as_tensor(qmap).detach().to("cpu", torch.float32).contiguous()
    if q.numel() != 256:
        raise ValueError(f"a map has 256 levels, not {q.numel()}")
    out = ctypes.c_uint8()
    _check(lib().bnb8_qmap_code(q.data_ptr(), float(x), ctypes.byref(out)))
    return int(out.value)


def bnb8_quantize_blockwise(x, qmap, blocksize: int = 256, codes=None, absmax=None, stream=None):
    torch = _torch()
    n = x.numel()
    nb = (n + blocksize - 1) // blocksize
    if codes is None:
        codes = torch.empty(n, dtype=torch.uint8, device=x.device)
    if absmax is None:
        absmax = torch.empty(nb, dtype=torch.float32, device=x.device)
    _check(lib().bnb8_quantize_blockwise(_ptr(x), _dtype_code(x), n, _ptr(qmap), blocksize,
                                         _ptr(codes), _ptr(absmax), _stream(stream)))
    return codes, absmax


def bnb8_dequantize_blockwise(codes, absmax, qmap, blocksize: int = 256, out=None, dtype=None,
                              stream=None):
    torch = _torch()
    if out is None:
        out = torch.empty(codes.numel(), dtype=dtype or torch.float32, device=codes.device)
    _check(lib().bnb8_dequantize_blockwise(_ptr(codes), _ptr(absmax), _ptr(qmap), blocksize,
                                           codes.numel(), _ptr(out), _dtype_code(out),
                                           _stream(stream)))
    return out


def bnb8_workspace_size(params: Sequence[ParamState], hp: HParams) -> int:
    if not params:
        return 0
    arr = _tensor_array(params)
    hc = hp.c(_dtype_code(params[0].p))
    return int(lib().bnb8_workspace_size(arr, len(params), ctypes.byref(hc)))


def _workspace(params, hp, workspace):
    torch = _torch()
    if hp.max_unorm == 0.0 and hp.blocksize != 0:
        return None, 0  # the step entry points need no workspace then
    need = bnb8_workspace_size(params, hp)
    if need == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=params[0].p.device)
    return workspace, workspace.numel()


def _step(entry: str, params, hp: HParams, qmap1, qmap2, workspace, stream):
    if not params:
        return
    arr = _tensor_array(params)
    hc = hp.c(_dtype_code(params[0].p))
    ws, ws_bytes = _workspace(params, hp, workspace)
    fn = getattr(lib(), entry)
    if entry == "bnb8_step_1state":
        _check(fn(arr, len(params), ctypes.byref(hc), _ptr(qmap1), _ptr(ws), ws_bytes,
                  _stream(stream)))
    else:
        _check(fn(arr, len(params), ctypes.byref(hc), _ptr(qmap1), _ptr(qmap2), _ptr(ws),
                  ws_bytes, _stream(stream)))


_ENTRY = {"adam": "bnb8_step_2state", "adamw": "bnb8_step_2state", "ademamix": "bnb8_step_ademamix",
          "momentum": "bnb8_step_1state", "rmsprop": "bnb8_step_1state",
          "adagrad": "bnb8_step_1state", "lion": "bnb8_step_1state"}


class Stepper:
    """The step entry point of hp.optim over a fixed tensor list, with the
    arguments marshalled once: the descriptor array, the hyperparameter
    struct, the workspace and the map pointers are built here, and each call
    only sets the update number and the stream.  The tensors (and the
    gradient tensors attached to them) must keep their storage while the
    Stepper is used."""

    def __init__(self, params, hp: HParams, qmap1, qmap2=None, workspace=None):
        self.n = len(params)
        self.arr = _tensor_array(params)
        self.hc = hp.c(_dtype_code(params[0].p)) if params else None
        self.ws, self.ws_bytes = _workspace(params, hp, workspace) if params else (None, 0)
        self.entry = _ENTRY[hp.optim]
        self.fn = getattr(lib(), self.entry)
        if self.entry == "bnb8_step_1state":
            self.args = (_ptr(qmap1), _ptr(self.ws), self.ws_bytes)
        else:
            self.args = (_ptr(qmap1), _ptr(qmap2), _ptr(self.ws), self.ws_bytes)
        self.hp_ref = ctypes.byref(self.hc) if params else None

    def __call__(self, step: int, stream=None):
        if self.n == 0:
            return
        self.hc.step = int(step)
        _check(self.fn(self.arr, self.n, self.hp_ref, *self.args, _stream(stream)))


def bnb8_step_2state(params, hp: HParams, qmap1, qmap2, workspace=None, stream=None):
    _step("bnb8_step_2state", params, hp, qmap1, qmap2, workspace, stream)


def bnb8_step_1state(params, hp: HParams, qmap1, workspace=None, stream=None):
    _step("bnb8_step_1state", params, hp, qmap1, None, workspace, stream)


def bnb8_step_ademamix(params, hp: HParams, qmap1, qmap2, workspace=None, stream=None):
    _step("bnb8_step_ademamix", params, hp, qmap1, qmap2, workspace, stream)


def bnb8_unorm(params, hp: HParams, qmap1, qmap2=None, out_scale=None, workspace=None,
               stream=None):
    torch = _torch()
    if out_scale is None:
        out_scale = torch.empty(len(params), dtype=torch.float32, device=params[0].p.device)
    arr = _tensor_array(params)
    hc = hp.c(_dtype_code(params[0].p))
    ws, ws_bytes = _workspace(params, hp, workspace)
    _check(lib().bnb8_unorm(arr, len(params), ctypes.byref(hc), _ptr(qmap1), _ptr(qmap2),
                            _ptr(out_scale), _ptr(ws), ws_bytes, _stream(stream)))
    return out_scale


def bnb8_unorm_static(params, hp: HParams, qmap1, qmap2=None, out_scale=None, stream=None):
    """bnb8_unorm without a workspace: for callers that cannot allocate device
    memory (the library's fixed 2 MiB scratch array holds the partial norms;
    at most 262,144 blocks per call; calls that overlap on the GPU race).
    out_scale (a float32 device tensor of len(params)) is required: this
    wrapper allocates nothing either."""
    if out_scale is None:
        raise ValueError("bnb8_unorm_static needs out_scale: it allocates no device memory")
    arr = _tensor_array(params)
    hc = hp.c(_dtype_code(params[0].p))
    _check(lib().bnb8_unorm_static(arr, len(params), ctypes.byref(hc), _ptr(qmap1), _ptr(qmap2),
                                   _ptr(out_scale), _stream(stream)))
    return out_scale


def step(params, hp: HParams, qmap1, qmap2=None, workspace=None, stream=None):
    """Dispatch to the entry point of hp.optim."""
    if hp.optim in ("adam", "adamw"):
        bnb8_step_2state(params, hp, qmap1, qmap2, workspace, stream)
    elif hp.optim == "ademamix":
        bnb8_step_ademamix(params, hp, qmap1, qmap2, workspace, stream)
    else:
        bnb8_step_1state(params, hp, qmap1, workspace, stream)


def split_blocks(ps: ParamState, blocksize: int, nchunks: int):
    """Split one tensor's descriptor into views at block boundaries.

    Blocks are quantized independently, so updating the pieces one by one is
    the same update as updating the whole tensor.  Works for the 1- and
    2-state layouts; AdEMAMix keeps m1 and m2 stacked as [2, n], which a view
    cannot split, so it is returned whole.  Returns (element ranges, pieces).
    """
    n = ps.p.numel()
    if ps.s1.numel() == 2 * n or blocksize == 0:
        # AdEMAMix keeps m1 and m2 stacked (8- or 32-bit); a tensor-wise
        # tensor is one block
        return [(0, n)], [ps]
    nb = (n + blocksize - 1) // blocksize
    per = max(1, -(-nb // max(1, nchunks)))
    ranges, pieces = [], []
    for b0 in range(0, nb, per):
        b1 = min(nb, b0 + per)
        lo, hi = b0 * blocksize, min(n, b1 * blocksize)
        cut = lambda t, a, b: None if t is None else t[a:b]
        g = cut(ps.g, lo, hi)
        if ps.state_bits == 8:
            piece = ParamState(ps.p[lo:hi], g, ps.s1[lo:hi], cut(ps.s2, lo, hi),
                               cut(ps.absmax1, b0, b1), cut(ps.absmax2, b0, b1), 8)
        else:
            piece = ParamState(ps.p[lo:hi], g, ps.s1[lo:hi], cut(ps.s2, lo, hi), None, None, 32)
        ranges.append((lo, hi))
        pieces.append(piece)
    return ranges, pieces


_ZERO_CODES = {}


def _zero_codes(optim: str, qmap1=None, qmap2=None):
    """(code of 0.0 under qmap1, under qmap2): maps default to the library's
    (bnb8_create_qmap: signed for s1 except RMSprop and Adagrad, unsigned for
    s2); the codes come from the library's nearest-level rule."""
    def code(q, signed):
        if q is not None:
            return bnb8_qmap_code(q, 0.0)
        if signed not in _ZERO_CODES:
            _ZERO_CODES[signed] = bnb8_qmap_code(bnb8_create_qmap(signed), 0.0)
        return _ZERO_CODES[signed]
    return code(qmap1, optim not in ("rmsprop", "adagrad")), code(qmap2, False)


def zero_state(p, optim: str, state_bits: int = 8, blocksize: int = 256, paged: bool = False,
               qmap1=None, qmap2=None):
    """Allocate the all-zero optimizer state of parameter p: every code is the
    code of 0.0 in its map (qmap1 / qmap2; by default the maps of
    bnb8_create_qmap the optimizer uses), every absmax 0.  blocksize 0:
    tensor-wise quantization, one absmax per state.  paged: the state arrays
    share one paged (managed) buffer (``paged_zero_states``)."""
    if paged:
        return paged_zero_states([(p, optim, state_bits, blocksize, qmap1, qmap2)])[0]
    torch = _torch()
    out = []
    zeros = _zero_codes(optim, qmap1, qmap2) if state_bits == 8 else (0, 0)
    for present, spec in _state_arrays(p.numel(), optim, state_bits, blocksize, zeros):
        if present is None:
            out.append(None)
            continue
        count, dtype, value = spec
        out.append(torch.full((count,), value, dtype=dtype, device=p.device))
    return tuple(out)


def _state_arrays(n: int, optim: str, state_bits: int, blocksize: int, zeros=(0, 0)):
    """(s1, s2, absmax1, absmax2) of an n-element parameter as
    (present, (count, dtype, zero value)) pairs; zeros = the codes of 0.0 of
    s1 and s2 (8-bit state)."""
    torch = _torch()
    k = NSTATES[optim]
    m = 2 if optim == "ademamix" else 1
    if state_bits == 32:
        return [(1, (n * m, torch.float32, 0.0)), (1 if k >= 2 else None, (n, torch.float32, 0.0)),
                (None, None), (None, None)]
    nb = 1 if blocksize == 0 else (n + blocksize - 1) // blocksize  # 0: tensor-wise
    two = 1 if k >= 2 else None
    return [(1, (n * m, torch.uint8, zeros[0])), (two, (n, torch.uint8, zeros[1])),
            (1, (nb * m, torch.float32, 0.0)), (two, (nb, torch.float32, 0.0))]


# ---- paged state -----------------------------------------------------------------

class _PagedBuffer:
    """One bnb8_paged_alloc buffer, exposed through the CUDA array interface:
    torch.as_tensor wraps it without a copy and holds a reference to this
    object for the tensor's lifetime; the buffer is freed with the last
    reference."""

    def __init__(self, count: int, dtype):
        torch = _torch()
        esize = torch.empty((), dtype=dtype).element_size()
        typestr = {torch.uint8: "|u1", torch.float32: "<f4", torch.float16: "<f2"}.get(dtype)
        if typestr is None:
            raise ValueError(f"paged buffers hold uint8, float32 or float16, not {dtype}")
        self.ptr = None
        ptr = ctypes.c_void_p()
        _check(lib().bnb8_paged_alloc(max(count * esize, 1), ctypes.byref(ptr)))
        self.ptr = ptr.value
        self.__cuda_array_interface__ = {"shape": (count,), "typestr": typestr,
                                         "data": (self.ptr, False), "version": 2}

    def __del__(self):
        if self.ptr:
            try:
                lib().bnb8_paged_free(self.ptr)
            except Exception:  # interpreter teardown: the process frees it
                pass


def paged_empty(count: int, dtype, device=None):
    """A 1-D tensor of ``count`` elements in paged memory (bnb8_paged_alloc):
    CUDA managed memory that the driver pages between host and device under
    device-memory pressure.  It behaves as an ordinary CUDA tensor of
    ``device``; contents are undefined."""
    torch = _torch()
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else \
        torch.device(device)
    with torch.cuda.device(device):
        buf = _PagedBuffer(int(count), dtype)
        return torch.as_tensor(buf, device=device)


def paged_zero_states(specs):
    """All-zero optimizer states (as ``zero_state``) of several parameters in
    ONE paged buffer: specs is a list of (p, optim, state_bits, blocksize),
    all p on one device; returns a list of (s1, s2, absmax1, absmax2), each
    array a 256-byte aligned slice of the shared buffer, so that one
    ``paged_prefetch`` call moves the states of all these parameters.  A spec
    may add (qmap1, qmap2) as in ``zero_state``."""
    torch = _torch()
    if not specs:
        return []
    device = specs[0][0].device
    layout, off = [], 0
    for spec_in in specs:
        p, optim, bits, blocksize = spec_in[:4]
        qm1, qm2 = (tuple(spec_in[4:6]) + (None, None))[:2]
        if p.device != device:
            raise ValueError("paged_zero_states: parameters on different devices")
        entry = []
        zeros = _zero_codes(optim, qm1, qm2) if bits == 8 else (0, 0)
        for present, spec in _state_arrays(p.numel(), optim, bits, blocksize, zeros):
            if present is None:
                entry.append(None)
                continue
            count, dtype, value = spec
            nbytes = count * torch.empty((), dtype=dtype).element_size()
            entry.append((off, count, dtype, value))
            off += (nbytes + 255) // 256 * 256
        layout.append(entry)
    arena = paged_empty(max(off, 256), torch.uint8, device)
    out = []
    for entry in layout:
        arrays = []
        for e in entry:
            if e is None:
                arrays.append(None)
                continue
            o, count, dtype, value = e
            esize = torch.empty((), dtype=dtype).element_size()
            arrays.append(arena[o:o + count * esize].view(dtype).fill_(value))
        out.append(tuple(arrays))
    return out


def paged_prefetch(tensors, device=None, stream=None) -> None:
    """Migrate paged memory (asynchronously, on ``stream``) to CUDA device
    ``device`` (default: the tensors' device) or, for ``"cpu"``, to host
    memory (bnb8_paged_prefetch).  ``tensors`` is one tensor or a list (None
    entries are skipped); each paged buffer they lie in is moved once, whole:
    the states that ``paged_zero_states`` packs together take one call."""
    torch = _torch()
    if torch.is_tensor(tensors):
        tensors = [tensors]
    seen = set()
    for t in tensors:
        if t is None:
            continue
        st = t.untyped_storage()
        if st.data_ptr() in seen:
            continue
        seen.add(st.data_ptr())
        if device is not None and torch.device(device).type == "cpu":
            dev = BNB8_PAGED_HOST
        else:
            dev = (t.device if device is None else torch.device(device)).index
            dev = torch.cuda.current_device() if dev is None else dev
        _check(lib().bnb8_paged_prefetch(st.data_ptr(), st.nbytes(), dev, _stream(stream)))
