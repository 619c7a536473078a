"""Helpers shared by the GPU parity tests: move numpy arrays (the oracle's
representation) to torch device tensors and back, run the same update on the
CUDA library and on the oracle, and compare."""
from __future__ import annotations

import numpy as np

import oracle

TORCH_DT = {"f32": "float32", "bf16": "bfloat16", "f16": "float16"}


def to_dev(a: np.ndarray, dtype: str | None = None, device="cuda"):
    """numpy -> torch on the device.  dtype names the storage of a uint16
    array (bf16 / f16 bit patterns)."""
    import torch
    if a is None:
        return None
    if dtype in ("bf16", "f16"):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
        t = t.view(torch.bfloat16 if dtype == "bf16" else torch.float16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(device)


def to_host(t) -> np.ndarray:
    import torch
    if t is None:
        return None
    t = t.detach().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def maps():
    return oracle.create_qmap(True), oracle.create_qmap(False)


def map_pair(optim: str, S: np.ndarray, U: np.ndarray):
    """(qmap1, qmap2) for an optimizer: signed first moments, unsigned second
    moments; RMSprop and Adagrad keep a non-negative single state."""
    if optim in ("adam", "adamw", "ademamix"):
        return S, U
    if optim in ("rmsprop", "adagrad"):
        return U, None
    return S, None


def random_state(optim: str, n: int, bits: int, B: int, seed: int, q1, q2):
    """A valid, non-trivial optimizer state (seeded)."""
    import workloads
    k = oracle.NSTATES[optim]
    m = 2 if optim == "ademamix" else 1
    if bits == 32:
        s1 = workloads.normal(n * m, 1e-3, seed)
        if optim in ("rmsprop", "adagrad"):
            s1 = np.abs(s1)
        s2 = np.abs(workloads.normal(n, 1e-6, seed + 1)) if k >= 2 else None
        return s1, s2, None, None
    nb = (n + B - 1) // B
    s1 = workloads.random_codes(n * m, seed)
    a1 = workloads.random_absmax(nb * m, 1e-3, seed + 1)
    s2 = a2 = None
    if k >= 2:
        s2 = workloads.random_codes(n, seed + 2)
        a2 = workloads.random_absmax(nb, 1e-6, seed + 3)
    return s1, s2, a1, a2


def assert_same(name, got: np.ndarray, want: np.ndarray):
    if got is None and want is None:
        return
    assert got.shape == want.shape, (name, got.shape, want.shape)
    if got.dtype == np.float32:
        gb, wb = got.view(np.uint32), want.view(np.uint32)
    else:
        gb, wb = got, want
    bad = np.nonzero(gb != wb)[0]
    if bad.size:
        i = bad[0]
        raise AssertionError(f"{name}: {bad.size} of {got.size} differ; first at {i}: "
                             f"got {got[i]!r} want {want[i]!r}")


def sample_blocks(n: int, B: int, count: int, seed: int):
    """Sorted distinct block indices: the first, the last and `count` random."""
    nb = (n + B - 1) // B
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(nb, size=min(count, nb), replace=False).tolist())
    pick.update({0, nb - 1})
    return sorted(pick)


def gather(t, blocks, B: int, n: int, base: int = 0, dtype: str | None = None):
    """Concatenate the elements of the given blocks of a device tensor (the
    stream starting at element `base`, of logical length n) on the host."""
    import torch
    idx = []
    for b in blocks:
        lo, hi = b * B, min(n, (b + 1) * B)
        idx.append(torch.arange(base + lo, base + hi, device=t.device))
    sel = t[torch.cat(idx)]
    return to_host(sel)


def gather_absmax(a, blocks, nblocks: int, base_block: int = 0):
    import torch
    sel = a[torch.tensor([base_block + b for b in blocks], device=a.device)]
    return to_host(sel)
