"""Seeded synthetic inputs for the 8-bit block-wise optimizer step.

This module only draws random numbers and describes shapes: it holds none of
the optimizer's arithmetic, so both the GPU library's tests/benchmark and the
CPU oracle can take their inputs from it.

Workloads (the shapes and value distributions of the method's own benchmark
and of large-model parameter lists):
  * ``adam_small``      one float32 tensor of 65,536 elements, p ~ N(0, 0.02),
                        g ~ N(0, 1e-3) drawn fresh each step.
  * ``adam_4096``       one 4096 x 4096 float32 tensor (16,777,216 elements),
                        g ~ N(0, 1e-3) with 1% of elements (Bernoulli mask)
                        drawn from N(0, 1e-1) as heavy-tail outliers.
  * ``embedding_rows``  a 50,257 x 1,024 bfloat16 tensor whose gradient is
                        exactly zero on 90% of rows (a seeded permutation picks
                        the 10% live rows, g ~ N(0, 1e-3) there).
  * ``dense_64m``       67,108,864 dense elements.
  * ``gpt2_xl_params``  the parameter-tensor shapes of a GPT-2-XL-sized model
                        (48 layers, d_model 1600, d_ff 6400, vocab 50,257,
                        1,024 positions, tied output head): 580 tensors,
                        1,557,611,200 elements.  No weights, only shapes.

Host arrays come from numpy's PCG64 (``np.random.default_rng(seed)``); device
tensors from a seeded torch generator on the device (used where host
generation of hundreds of millions of values would dominate a run).
"""
from __future__ import annotations

import numpy as np

# ---- host (numpy) generators -------------------------------------------------


def normal(n: int, std: float, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(n, dtype=np.float32) * np.float32(std)).astype(np.float32)


def normal_with_outliers(n: int, std: float, outlier_std: float, outlier_frac: float,
                         seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(n, dtype=np.float32) * np.float32(std)
    mask = rng.random(n) < outlier_frac
    x[mask] = rng.standard_normal(int(mask.sum()), dtype=np.float32) * np.float32(outlier_std)
    return x.astype(np.float32)


def sparse_rows(rows: int, cols: int, live_frac: float, std: float, seed: int) -> np.ndarray:
    """Row-sparse gradient: ``live_frac`` of rows N(0, std), the rest exactly 0."""
    rng = np.random.default_rng(seed)
    live = rng.permutation(rows)[: int(round(rows * live_frac))]
    g = np.zeros((rows, cols), dtype=np.float32)
    g[live] = rng.standard_normal((live.size, cols), dtype=np.float32) * np.float32(std)
    return g.reshape(-1)


def random_codes(n: int, seed: int) -> np.ndarray:
    return np.random.default_rng(seed).integers(0, 256, n, dtype=np.uint8)


def random_absmax(nblocks: int, scale: float, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return (np.abs(rng.standard_normal(nblocks, dtype=np.float32)) * np.float32(scale)
            + np.float32(scale * 1e-3)).astype(np.float32)


# ---- device (torch) generators ---------------------------------------------


def torch_normal(n: int, std: float, seed: int, device, dtype=None):
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    x = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
    x.mul_(std)
    return x if dtype is None else x.to(dtype)


def torch_normal_with_outliers(n: int, std: float, outlier_std: float, outlier_frac: float,
                               seed: int, device, dtype=None):
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    x = torch.randn(n, generator=gen, device=device, dtype=torch.float32).mul_(std)
    mask = torch.rand(n, generator=gen, device=device) < outlier_frac
    out = torch.randn(n, generator=gen, device=device, dtype=torch.float32).mul_(outlier_std)
    x = torch.where(mask, out, x)
    return x if dtype is None else x.to(dtype)


def torch_sparse_rows(rows: int, cols: int, live_frac: float, std: float, seed: int, device,
                      dtype=None):
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    live = torch.randperm(rows, generator=gen, device=device)[: int(round(rows * live_frac))]
    g = torch.zeros(rows, cols, device=device, dtype=torch.float32)
    g[live] = torch.randn(live.numel(), cols, generator=gen, device=device).mul_(std)
    g = g.reshape(-1)
    return g if dtype is None else g.to(dtype)


def torch_random_codes(n: int, seed: int, device):
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return torch.randint(0, 256, (n,), generator=gen, device=device, dtype=torch.int32).to(
        torch.uint8)


def torch_random_absmax(nblocks: int, scale: float, seed: int, device):
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    x = torch.randn(nblocks, generator=gen, device=device, dtype=torch.float32).abs_()
    return x.mul_(scale).add_(scale * 1e-3)


# ---- shapes ------------------------------------------------------------------


def gpt2_xl_params(n_layer: int = 48, d: int = 1600, d_ff: int = 6400, vocab: int = 50257,
                   n_pos: int = 1024):
    """(name, numel) of every parameter tensor of a GPT-2-XL-shaped model."""
    shapes = [("wte", vocab * d), ("wpe", n_pos * d)]
    for i in range(n_layer):
        pre = f"h{i}."
        shapes += [
            (pre + "ln_1.weight", d), (pre + "ln_1.bias", d),
            (pre + "attn.c_attn.weight", d * 3 * d), (pre + "attn.c_attn.bias", 3 * d),
            (pre + "attn.c_proj.weight", d * d), (pre + "attn.c_proj.bias", d),
            (pre + "ln_2.weight", d), (pre + "ln_2.bias", d),
            (pre + "mlp.c_fc.weight", d * d_ff), (pre + "mlp.c_fc.bias", d_ff),
            (pre + "mlp.c_proj.weight", d_ff * d), (pre + "mlp.c_proj.bias", d),
        ]
    shapes += [("ln_f.weight", d), ("ln_f.bias", d)]
    return shapes
