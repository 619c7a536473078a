"""Benchmark of the 8-bit block-wise optimizer step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one optimizer update (one call of the library's step entry point)
over the workload's synthetic parameters and gradients, which are resident in
HBM before timing starts.  W untimed warm-up steps, then exactly K timed steps
bracketed by a barrier and a device synchronize; the L2 cache is flushed before
every timed step (256 MiB written, then 256 MiB of other data read, so the
step starts with clean, unrelated lines) and each step is timed with CUDA
events on the launching stream.  Rank 0 prints one JSON line.

Under torchrun (N > 1) every rank runs its own full replica of the workload
on its own GPU (blocks are independent units with no exchange step), so the
whole-job value is the units all ranks processed over the slowest rank's
time ("scaling": "weak").

--impl reference times the CPU oracle (the single-threaded C statement of the
method) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "Gelem/s per optimizer step and achieved HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "Gelem/s"
L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 129 << 20            # GB300 L2 (about 126 MiB)
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
class Workload:
    """A tensor list, its dtype, optimizer and hyperparameters, and the
    algorithmic bytes one step must move (reads + writes of p, g, the state
    codes / values and the per-block absmax; the 2 KB of maps are ignored).
    op "quantize" / "dequantize": the stand-alone block-wise conversion of
    one tensor instead of an optimizer step.
    paged "resident": the states live in paged (managed) memory and every step
    prefetches them to the device first, as the paged optimizers do; "evicted":
    the same, with the states paged out to the host before every step (outside
    the timed region), so that each timed step migrates them back."""

    def __init__(self, name, desc, optim, dtype, sizes, bits, blocksize, hp, grad, p_std=0.02,
                 op="step", paged=None, carry=False, pages=None):
        self.name, self.desc, self.optim, self.dtype = name, desc, optim, dtype
        self.sizes, self.bits, self.blocksize, self.hp = sizes, bits, blocksize, hp
        self.grad, self.p_std, self.op, self.paged = grad, p_std, op, paged
        self.carry = carry   # ||p|| carried between steps (BNB8_CARRY_PNORM)
        # the pages' own figure for this workload, as (ms per step, source), or None
        self.pages = pages

    def lib_hp(self):
        """Keyword arguments of the library's HParams (the oracle's plus the
        carried-norm switch, which changes no result's definition)."""
        return dict(self.hp, carry_pnorm=self.carry)

    @property
    def elements(self):
        return int(sum(self.sizes))

    def nstates(self):
        return {"adam": 2, "adamw": 2, "ademamix": 3}.get(self.optim, 1)

    def read_bytes(self):
        """Bytes a step reads (p, g, states, absmax): what must exceed the L2
        for back-to-back steps to find none of their inputs there."""
        e = 4 if self.dtype == "f32" else 2
        ns, B = self.nstates(), self.blocksize
        total = 0
        for n, b in zip(self.sizes, self.bits):
            nb = 1 if B == 0 else (n + B - 1) // B
            total += 2 * n * e + (n * ns + nb * 4 * ns if b == 8 else n * 4 * ns)
        return total

    def algorithmic_bytes(self, live_block_frac=1.0):
        e = 4 if self.dtype == "f32" else 2
        if self.op != "step":
            # read x, write codes + absmax (quantize), or the reverse
            n, nb = self.elements, -(-self.elements // self.blocksize)
            return int(n * e + n + nb * 4)
        ns, B = self.nstates(), self.blocksize
        total = 0.0
        for n, b in zip(self.sizes, self.bits):
            nb = 1 if B == 0 else (n + B - 1) // B
            if b == 8 and B == 0:
                # tensor-wise: a first pass reads p, g and the codes for the
                # new absmax, the second is the step
                total += n * 2 * e + n * ns
            if b == 8:
                rest = n * (2 * e + 2 * ns) + nb * 8 * ns  # p r+w, codes r+w, absmax r+w
            else:
                rest = n * (2 * e + 8 * ns)                # p r+w, binary32 states r+w
            total += n * e + rest * live_block_frac        # g always read
            if self.hp.get("max_unorm", 0.0) > 0 and not self.hp.get("unorm_per_block"):
                # the per-tensor pre-pass reads g, p, states (per block: inside
                # the step); with the norm carried from the previous step it
                # reads p only when the direction needs it (coupled decay)
                decoupled = self.optim in ("adamw", "lion", "ademamix")
                p_read = not (self.carry and (decoupled or self.hp.get("weight_decay", 0.0) == 0))
                total += n * e * (2 if p_read else 1) + \
                    (n * ns + nb * 4 * ns if b == 8 else n * 4 * ns)
        return int(total)


_HP_1STATE = {"momentum": dict(lr=0.01, beta1=0.9), "rmsprop": dict(lr=0.01, beta1=0.99),
              "adagrad": dict(lr=0.01), "lion": dict(lr=1e-4, beta1=0.9, beta2=0.99),
              "adam": dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)}


def _cfg_embedding(optim, skip):
    name = {"momentum": "Momentum", "rmsprop": "RMSprop", "adagrad": "Adagrad", "lion": "Lion",
            "adam": "Adam"}[optim]
    return Workload(
        f"{optim}8bit_50257x1024_bf16_B256_rowsparse_{'skipzeros' if skip else 'noskip'}",
        f"{name}8bit on a 50,257 x 1,024 bf16 embedding, 90% of gradient rows exactly zero, "
        f"skip_zeros {'on' if skip else 'off'}",
        optim, "bf16", [50257 * 1024], [8], 256, dict(_HP_1STATE[optim], skip_zeros=skip),
        ("rows", 50257, 1024, 0.1, 1e-3))


def _cfg_dense_1state(optim):
    name = {"rmsprop": "RMSprop", "adagrad": "Adagrad"}[optim]
    return Workload(f"{optim}8bit_64M_bf16_B256", f"{name}8bit, 67,108,864 dense bf16",
                    optim, "bf16", [1 << 26], [8], 256, dict(_HP_1STATE[optim]),
                    ("normal", 1e-3))


def _cfg_codec(op):
    n = 4096 * 4096
    what = ("float32 -> uint8 codes + absmax" if op == "quantize"
            else "uint8 codes + absmax -> float32")
    return Workload(f"{op}_blockwise_4096x4096_f32_B256",
                    f"stand-alone block-wise {op} of one 4096x4096 tensor ({what}), block 256, "
                    f"signed dynamic map, x ~ N(0,1e-3) with 1% N(0,1e-1) outliers",
                    "adam", "f32", [n], [8], 256, {}, ("outliers", 1e-3, 1e-1, 0.01), op=op)


def _cfg_unorm(per_block):
    n = 4096 * 4096
    how = "per block (inside the step)" if per_block else "per tensor (pre-pass + step)"
    return Workload(
        f"adam8bit_4096x4096_f32_B256_maxunorm_{'block' if per_block else 'tensor'}",
        f"Adam8bit blockwise, one 4096x4096 float32 tensor, block 256, max_unorm 0.5 {how}, "
        f"g ~ N(0,1e-3) with 1% N(0,1e-1) outliers, wd 1e-2",
        "adam", "f32", [n], [8], 256,
        dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=1e-2, max_unorm=0.5,
             unorm_per_block=per_block),
        ("outliers", 1e-3, 1e-1, 0.01))


def _cfg_adam_4096(optim="adam", B=256):
    n = 4096 * 4096
    kind = f"blockwise, block {B}" if B else "tensor-wise (one absmax per state per tensor)"
    return Workload(
        f"{optim}8bit_4096x4096_f32_{'B%d' % B if B else 'tensorwise'}",
        f"{'Adam' if optim == 'adam' else 'AdamW'}8bit {kind}, one 4096x4096 float32 tensor "
        f"(16,777,216 elements), g ~ N(0,1e-3) with 1% N(0,1e-1) outliers, wd 1e-2",
        optim, "f32", [n], [8], B,
        dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=1e-2),
        ("outliers", 1e-3, 1e-1, 0.01))


# "[XPU] Implemented 8bit optimizers in triton #1692": the 8-bit step of the
# fused Triton kernel on one 4096x4096 bf16 tensor with grads randn * 0.01 took
# 1.250-1.325 ms on an Intel Data Center GPU Max 1100 (another machine: context).
# The posted script selects the AdEMAMix 8-bit blockwise optimizer while the
# text speaks of an Adam-family step, so both are run.
PAGES_4096_BF16_MS = (1.250 + 1.325) / 2


def _cfg_pages_4096(optim):
    n = 4096 * 4096
    name = {"adam": "Adam", "ademamix": "AdEMAMix"}[optim]
    return Workload(
        f"{optim}8bit_4096x4096_bf16_B256_pages_workload",
        f"{name}8bit blockwise, one 4096x4096 bf16 tensor, block 256, bf16 grads ~ N(0, 1e-2) "
        "(the PR #1692 benchmark's shape and gradients)", optim, "bf16", [n], [8], 256,
        dict(HP_PAGES[optim]), ("normal", 1e-2),
        pages=(PAGES_4096_BF16_MS, "[XPU] Implemented 8bit optimizers in triton #1692: "
               "1.250-1.325 ms per step on an Intel Data Center GPU Max 1100 (another machine)"))


HP_PAGES = {"adam": dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8),
            "ademamix": dict(lr=1e-3, beta1=0.9, beta2=0.999, beta3=0.9999, alpha=5.0, eps=1e-8)}


def _cfg_paged(mode):
    n = 4096 * 4096
    how = ("resident, prefetched to the device before every step" if mode == "resident" else
           "paged out to the host before every step, migrated back inside the timed step")
    return Workload(
        f"adam8bit_4096x4096_f32_B256_paged_{mode}",
        f"PagedAdam8bit blockwise, one 4096x4096 float32 tensor, block 256, states in paged "
        f"(managed) memory {how}, g ~ N(0,1e-3) with 1% N(0,1e-1) outliers, wd 1e-2",
        "adam", "f32", [n], [8], 256,
        dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=1e-2),
        ("outliers", 1e-3, 1e-1, 0.01), paged=mode)


def _cfg_gpt2xl(optim="adam", carry=False):
    shapes = workloads.gpt2_xl_params()
    sizes = [n for _, n in shapes]
    bits = [8 if n >= 4096 else 32 for n in sizes]
    name = "Adam" if optim == "adam" else "AdamW"
    return Workload(f"gpt2xl_list_bf16_{optim}8bit_B256_maxunorm1{'_carried' if carry else ''}",
                    "GPT-2-XL-shaped list (580 tensors, 1,557,611,200 elements), bf16 p/g, "
                    f"tensors < 4096 elements at 32-bit state, {name}8bit B256, max_unorm 1.0, "
                    f"wd 0.1{', ||p|| carried from the previous step' if carry else ''}",
                    optim, "bf16", sizes, bits, 256,
                    dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1,
                         max_unorm=1.0), ("normal", 1e-3), carry=carry)


WORKLOADS = {
    "adam_4096": lambda: _cfg_adam_4096("adam", 256),
    "adamw_4096": lambda: _cfg_adam_4096("adamw", 256),
    "adam_4096_b2048": lambda: _cfg_adam_4096("adam", 2048),
    "adam_small": lambda: Workload("adam8bit_65536_f32_B256", "Adam8bit, one 65,536-element "
                                   "float32 tensor, block 256", "adam", "f32", [65536], [8], 256,
                                   dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8),
                                   ("normal", 1e-3)),
    "momentum_embedding": lambda: Workload(
        "momentum8bit_50257x1024_bf16_B256_rowsparse_skipzeros",
        "Momentum8bit on a 50,257 x 1,024 bf16 embedding, 90% of gradient rows exactly zero, "
        "skip_zeros", "momentum", "bf16", [50257 * 1024], [8], 256,
        dict(lr=0.01, beta1=0.9, skip_zeros=True), ("rows", 50257, 1024, 0.1, 1e-3)),
    "lion_64m": lambda: Workload("lion8bit_64M_bf16_B256", "Lion8bit, 67,108,864 dense bf16",
                                 "lion", "bf16", [1 << 26], [8], 256,
                                 dict(lr=1e-4, beta1=0.9, beta2=0.99), ("normal", 1e-3)),
    "momentum_64m": lambda: Workload("momentum8bit_64M_bf16_B256",
                                     "Momentum8bit, 67,108,864 dense bf16", "momentum", "bf16",
                                     [1 << 26], [8], 256, dict(lr=0.01, beta1=0.9),
                                     ("normal", 1e-3)),
    "ademamix_64m": lambda: Workload("ademamix8bit_64M_f32_B256",
                                     "AdEMAMix8bit, 67,108,864 float32, alpha 5, betas "
                                     "(0.9, 0.999, 0.9999), t_alpha = t_beta3 = 100",
                                     "ademamix", "f32", [1 << 26], [8], 256,
                                     dict(lr=1e-3, beta1=0.9, beta2=0.999, beta3=0.9999,
                                          alpha=5.0, t_alpha=100, t_beta3=100, eps=1e-8),
                                     ("normal", 1e-3)),
    "gpt2xl": _cfg_gpt2xl,
    "gpt2xl_carried": lambda: _cfg_gpt2xl("adam", True),
    "gpt2xl_adamw": lambda: _cfg_gpt2xl("adamw"),
    "gpt2xl_adamw_carried": lambda: _cfg_gpt2xl("adamw", True),
    **{f"{o}_embedding{sfx}": (lambda o=o, sk=sk: _cfg_embedding(o, sk))
       for o in ("momentum", "rmsprop", "adagrad", "lion", "adam") for sfx, sk in (("", True), ("_noskip", False))
       if not (o == "momentum" and sk)},
    **{f"{o}_64m": (lambda o=o: _cfg_dense_1state(o)) for o in ("rmsprop", "adagrad")},
    "adam_4096_tensorwise": lambda: _cfg_adam_4096(B=0),
    "adam_4096_bf16_pages": lambda: _cfg_pages_4096("adam"),
    "ademamix_4096_bf16_pages": lambda: _cfg_pages_4096("ademamix"),
    "adam_4096_paged": lambda: _cfg_paged("resident"),
    "adam_4096_paged_evicted": lambda: _cfg_paged("evicted"),
    "adamw_4096_b2048": lambda: _cfg_adam_4096("adamw", 2048),
    "quantize_4096": lambda: _cfg_codec("quantize"),
    "dequantize_4096": lambda: _cfg_codec("dequantize"),
    "adam_4096_unorm": lambda: _cfg_unorm(False),
    "adam_4096_unorm_block": lambda: _cfg_unorm(True),
}
DEFAULT_WORKLOAD = "adam_4096"


# The host enqueues the timed steps ahead of the device: every
# HOST_AHEAD_STEPS steps a sleep kernel of HOST_AHEAD_US_PER_STEP per step
# (outside every event pair) gives the host the time to queue the next ones.
HOST_AHEAD_STEPS = 25
HOST_AHEAD_US_PER_STEP = 150.0


def gpu_sleep(stream, us):
    """Keep `stream` busy for about `us` microseconds (torch's spin kernel)."""
    import torch
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is None:
        return
    with torch.cuda.stream(stream):
        sleep(int(us * 2000))  # cycles at about 2 GHz


def step_distribution(per_step_ms):
    """Median, mean, p10 and p90 of the per-step event times (ms)."""
    xs = sorted(per_step_ms)
    k = len(xs)
    pick = lambda q: xs[min(k - 1, max(0, int(round(q * (k - 1)))))]
    return {"median": statistics.median(xs), "mean": sum(xs) / k, "p10": pick(0.1),
            "p90": pick(0.9), "min": xs[0], "max": xs[-1]}


def _device_grad(wl, n, seed, device, torch_dtype):
    kind = wl.grad[0]
    if kind == "outliers":
        return workloads.torch_normal_with_outliers(n, wl.grad[1], wl.grad[2], wl.grad[3], seed,
                                                    device, torch_dtype)
    if kind == "rows":
        return workloads.torch_sparse_rows(wl.grad[1], wl.grad[2], wl.grad[3], wl.grad[4], seed,
                                           device, torch_dtype)
    return workloads.torch_normal(n, wl.grad[1], seed, device, torch_dtype)


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
CLOCK_FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, uuid=None, period_ms=20):
        self.path = tempfile.mktemp(prefix="bnb8_clocks_", suffix=".csv")
        cmd = ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
               f"-lms={period_ms}"]
        if uuid:
            cmd.insert(1, f"--id={uuid}")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append(dict(t=ts, sm=float(parts[1]), sm_max=float(parts[2]),
                                     power=parts[3], hw=parts[5], hw_thermal=parts[6],
                                     sw_thermal=parts[7], sw_power=parts[8]))
                except ValueError:
                    continue
        os.unlink(self.path)
        return rows


def summarize_clocks(rows, t0, t1):
    inside = [r for r in rows if t0 - 0.05 <= r["t"] <= t1 + 0.05] or rows
    if not inside:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    reasons = set()
    for r in inside:
        for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                          ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
            if r[key].lower().startswith("active"):
                reasons.add(name)
    return {"sm_mhz": statistics.median(r["sm"] for r in inside),
            "sm_max_mhz": max(r["sm_max"] for r in inside), "reasons": sorted(reasons),
            "samples": len(inside)}


# ---------------------------------------------------------------------------
# peaks and committed ncu traffic
# ---------------------------------------------------------------------------
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def vs_pages(wl, value):
    """value over the pages' own figure for this exact workload (another
    machine's number: context, not the target), or None when the pages give
    none for it."""
    if not wl.pages:
        return None
    pages_gelem = wl.elements / (wl.pages[0] * 1e-3) / 1e9
    return round(value / pages_gelem, 2)


def kernel_source_hash():
    """Hash of the device code (kernel files, device helpers, launch
    arguments): the host API can change without invalidating a capture."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_block_wise_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.startswith("k_") or name in ("bnb8_device.cuh", "bnb8_internal.h"):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload_name):
    """Per-launch DRAM bytes of the step kernel from the committed ncu summary,
    or None when it was taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload_name)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("kernel_source_hash") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def setup_dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def build_state(bnb8, wl, device, seed=0):
    import torch
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[wl.dtype]
    params = []
    for i, (n, b) in enumerate(zip(wl.sizes, wl.bits)):
        p = workloads.torch_normal(n, wl.p_std, seed + i, device, tdt)
        s1, s2, a1, a2 = bnb8.zero_state(p, wl.optim, b, wl.blocksize, paged=wl.paged is not None)
        params.append(bnb8.ParamState(p, None, s1, s2, a1, a2, b))
    return params, tdt


def run_gpu(args, wl):
    if wl.op != "step":
        return run_codec(args, wl)
    import torch
    import bit_block_wise_gb300 as bnb8
    from bit_block_wise_gb300 import build as bnb8_build

    world, rank, local = setup_dist()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    bnb8_build.build()
    stream = torch.cuda.current_stream()
    q1 = bnb8.bnb8_create_qmap(wl.optim not in ("rmsprop", "adagrad")).to(device)
    q2 = bnb8.bnb8_create_qmap(False).to(device)
    params, tdt = build_state(bnb8, wl, device, seed=1000 * rank)
    # a pool of gradients (fresh g every step, all resident before timing)
    pool = 2 if wl.elements > (1 << 28) else 4
    grads = [[_device_grad(wl, n, 7919 * (k + 1) + i + 100000 * rank, device, tdt)
              for i, n in enumerate(wl.sizes)] for k in range(pool)]
    hp_kw = dict(wl.hp)
    ws_bytes = bnb8.bnb8_workspace_size(params, bnb8.HParams(optim=wl.optim, blocksize=wl.blocksize,
                                                             **hp_kw))
    workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    flush_read = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)
    flush_sink = torch.empty((), dtype=torch.int32, device=device)

    def flush_l2():
        # write more than the L2 holds, then read as much other data (a max
        # reduction: it keeps the dtype, so it writes no temporary): the L2
        # ends up holding clean lines of unrelated buffers, so the timed step
        # neither hits its own data nor pays for the flush's write-backs
        flush.zero_()
        torch.amax(flush_read, 0, out=flush_sink)

    step_no = [0]
    state_arrays = [t for ps in params for t in (ps.s1, ps.s2, ps.absmax1, ps.absmax2)
                    if t is not None]
    # Between timed steps: flush the L2, or (inputs well over the L2's size)
    # run the steps back to back: each then starts with the lines the last
    # one left, dirty ones included, and none of its own inputs
    l2_mode = args.l2
    if l2_mode == "auto":
        l2_mode = "none" if wl.read_bytes() >= 1.2 * L2_BYTES and not wl.paged else "flush"
    if l2_mode == "none" and wl.read_bytes() < 1.2 * L2_BYTES:
        l2_mode = "flush"

    def page_out():
        # device-memory pressure elsewhere has moved the states to the host
        if wl.paged == "evicted":
            bnb8.paged_prefetch(state_arrays, "cpu", stream)

    # the library's marshal-once entry (Stepper), one per gradient set of the
    # pool: inside the timed region a step is one ctypes call
    hp0 = bnb8.HParams(optim=wl.optim, blocksize=wl.blocksize, step=1, **wl.lib_hp())
    steppers = []
    for k in range(pool):
        for ps, g in zip(params, grads[k]):
            ps.g = g
        steppers.append(bnb8.Stepper(params, hp0, q1, q2,
                                     workspace=workspace if ws_bytes else None))

    def one_step(k):
        step_no[0] += 1
        if wl.paged is not None:
            bnb8.paged_prefetch(state_arrays, device, stream)  # one call per paged buffer
        steppers[k % pool](step_no[0], stream)

    for k in range(args.warmup):
        page_out()
        one_step(k)
    torch.cuda.synchronize()

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid) if rank == 0 else None
    time.sleep(0.3 if sampler else 0.0)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    for k in range(args.steps):
        if k % HOST_AHEAD_STEPS == 0:
            # keep the device behind the host: a sleep kernel (outside the
            # timed region) covers the host's time to enqueue the next steps,
            # so no event pair ever waits for a launch
            gpu_sleep(stream, HOST_AHEAD_STEPS * HOST_AHEAD_US_PER_STEP)
        page_out()
        if l2_mode == "flush":
            flush_l2()
        starts[k].record(stream)
        one_step(args.warmup + k)
        ends[k].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    rows = sampler.stop() if sampler else []
    per_step = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    dist_ms = step_distribution(per_step)
    ms_per_step = max_over_ranks(dist_ms["median"], world, device)
    # the library's plan: at most 96 tensors per launch; 8-bit tensors that
    # are multiples of max(512, B) elements launch apart from the others
    # (every tensor here is 256-byte aligned)
    unit = max(512, wl.blocksize)
    whole8 = sum(1 for n, b in zip(wl.sizes, wl.bits) if b == 8 and n % unit == 0)
    rest8 = sum(1 for b in wl.bits if b == 8) - whole8
    n_chunks8 = -(-whole8 // 96) + -(-rest8 // 96)
    n_chunks32 = -(-sum(1 for b in wl.bits if b == 32) // 96)
    launches_per_step = n_chunks8 + n_chunks32
    if wl.hp.get("max_unorm", 0.0) > 0 and not wl.hp.get("unorm_per_block"):
        # per launch group: pre-pass, reduction (chunk sums and multipliers)
        launches_per_step += 2 * (n_chunks8 + n_chunks32)
    if wl.blocksize == 0:
        launches_per_step += 1 + 2 * n_chunks8                  # fill + absmax pass + store

    # ---- end to end through the public API with host buffers ----
    e2e = run_e2e(args, wl, bnb8, params, q1, q2, workspace, ws_bytes, stream, step_no, tdt)

    value = world * wl.elements / (ms_per_step * 1e-3) / 1e9
    alg_bytes = wl.algorithmic_bytes(live_frac(wl, grads[0]) if wl.hp.get("skip_zeros") else 1.0)
    achieved = alg_bytes / (ms_per_step * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    out = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "step_ms": {k: round(v, 5) for k, v in dist_ms.items()},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": vs_pages(wl, value),
        "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.desc, "name": wl.name, "elements": wl.elements,
                   "tensors": len(wl.sizes), "blocksize": wl.blocksize, "optimizer": wl.optim,
                   "param_dtype": wl.dtype, "arithmetic": "binary32",
                   "state": "uint8 codes + binary32 absmax",
                   "timing": "median of per-step CUDA event pairs on the launching stream; "
                             "the host enqueues ahead of the device",
                   "l2": ("flushed before every timed step (256 MiB written, then 256 MiB of "
                          "other data read, leaving clean unrelated lines)" if l2_mode == "flush"
                          else f"not flushed: the step reads {wl.read_bytes() / 2**20:.0f} MiB, "
                               f"more than the {L2_BYTES / 2**20:.0f} MiB L2; steps run back to "
                               "back, each starting with the previous one's lines (dirty ones "
                               "included)"),
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   **({"pages_figure": {"ms_per_step": wl.pages[0], "source": wl.pages[1]}}
                      if wl.pages else {})},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                     "algorithmic_bytes_per_step": alg_bytes,
                     "traffic": ncu_traffic(wl.name)},
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": summarize_clocks(rows, t0, t1),
    }
    if wl.paged:
        out["config"]["paged"] = {
            "mode": wl.paged,
            "state_bytes": int(sum(t.numel() * t.element_size() for t in state_arrays)),
            "migrated_host_to_device_in_timed_step": wl.paged == "evicted"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the CPU (oracle) leg: the timed baseline, then the oracle's check of
        # one more GPU step on sampled blocks (outside every timed region)
        out["cpu_baseline"] = cpu_baseline(wl, params, budget_s=args.cpu_budget)
        step_no[0] += 1
        out["parity_sample"] = sampled_parity(
            wl, params, lambda: steppers[0](step_no[0], stream), step_no[0], grads[0])
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def live_frac(wl, grads):
    """Fraction of blocks with a nonzero gradient (skip_zeros traffic model)."""
    import torch
    B = wl.blocksize
    live, total = 0, 0
    for g in grads:
        n = g.numel()
        nb = n // B
        if nb:
            live += int((g[: nb * B].view(nb, B) != 0).any(dim=1).sum().item())
            total += nb
    return live / max(total, 1)


def e2e_groups(bnb8, params, wl, ngroups):
    """Work of one step in about ngroups launches: tensors larger than a
    group's share are split at block boundaries (blocks are independent), and
    consecutive pieces are packed into groups of about equal size.  With
    max_unorm every tensor stays whole (its norm needs all of its blocks in
    one call).  Returns a list of groups, each a list of
    (tensor index, (lo, hi), piece)."""
    target = -(-wl.elements // ngroups)
    whole = (wl.hp.get("max_unorm", 0.0) > 0 and not wl.hp.get("unorm_per_block")) or \
        wl.blocksize == 0
    pieces = []
    for i, ps in enumerate(params):
        n = ps.p.numel()
        k = 1 if whole else max(1, -(-n // target))
        if k == 1:
            pieces.append((i, (0, n), ps))
        else:
            ranges, pcs = bnb8.split_blocks(ps, wl.blocksize, k)
            pieces += [(i, r, pc) for r, pc in zip(ranges, pcs)]
    groups, cur, size = [], [], 0
    for item in pieces:
        cur.append(item)
        size += item[1][1] - item[1][0]
        if size >= target:
            groups.append(cur)
            cur, size = [], 0
    if cur:
        groups.append(cur)
    return groups


def run_e2e(args, wl, bnb8, params, q1, q2, workspace, ws_bytes, stream, step_no, tdt):
    """The same step through the public API with the gradient arriving from
    pinned host memory and the updated parameter read back to pinned host
    memory, every step.  The work is cut into four launches of about equal
    size (e2e_groups), so that the upload of group i+1, the step on group i
    and the read-back of group i-1 run concurrently on three streams; each
    launch is a Stepper (arguments marshalled once).  The device gradient is
    double-buffered, so the next step's uploads start while this step's
    launches still read the other buffer and the link never drains."""
    import torch
    if wl.elements > (1 << 28):
        steps = max(2, min(args.steps, 5))
    else:
        steps = max(3, min(args.steps, 50))
    host_g = [torch.empty(n, dtype=tdt, pin_memory=True) for n in wl.sizes]
    host_p = [torch.empty(n, dtype=tdt, pin_memory=True) for n in wl.sizes]
    for hg, ps in zip(host_g, params):
        hg.copy_(ps.g if ps.g is not None else torch.zeros_like(ps.p))
    hp0 = bnb8.HParams(optim=wl.optim, blocksize=wl.blocksize, step=1, **wl.lib_hp())
    dev_g, groups, steppers = [], [], []
    # a carried norm lives in the workspace of its own tensor list: one per
    # group, shared by the group's two gradient buffers
    group_ws = {}

    def ws_for(c):
        if not ws_bytes:
            return None
        if not wl.carry:
            return workspace
        if c not in group_ws:
            group_ws[c] = torch.zeros_like(workspace)
        return group_ws[c]
    for buf in range(2):
        dev_g.append([torch.empty_like(ps.p) for ps in params])
        for ps, dg in zip(params, dev_g[buf]):
            ps.g = dg
        groups.append(e2e_groups(bnb8, params, wl, 4))
        steppers.append([bnb8.Stepper([pc for _, _, pc in grp], hp0, q1, q2, workspace=ws_for(c))
                         for c, grp in enumerate(groups[buf])])
    ngroups = len(groups[0])
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_up = [torch.cuda.Event() for _ in range(ngroups)]
    ev_done = [[torch.cuda.Event() for _ in range(ngroups)] for _ in range(2)]
    ev_back = [torch.cuda.Event() for _ in range(ngroups)]
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    for k in range(steps):
        step_no[0] += 1
        buf = k % 2
        for c, grp in enumerate(groups[buf]):
            with torch.cuda.stream(s_in):
                # this buffer's previous readers (two steps back) are done
                s_in.wait_event(ev_done[buf][c])
                for i, (lo, hi), _ in grp:
                    dev_g[buf][i][lo:hi].copy_(host_g[i][lo:hi], non_blocking=True)
                ev_up[c].record(s_in)
            stream.wait_event(ev_up[c])
            if k > 0:                           # p of this group is still being read back
                stream.wait_event(ev_back[c])
            steppers[buf][c](step_no[0], stream)
            ev_done[buf][c].record(stream)
            s_out.wait_event(ev_done[buf][c])
            with torch.cuda.stream(s_out):
                for i, (lo, hi), pc in grp:
                    host_p[i][lo:hi].copy_(pc.p, non_blocking=True)
                ev_back[c].record(s_out)
    s_out.wait_stream(s_in)
    s_out.wait_stream(stream)
    end.record(s_out)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    esz = 4 if wl.dtype == "f32" else 2
    return {"value": round(wl.elements / (ms * 1e-3) / 1e9, 3), "unit": UNIT,
            "h2d_bytes_per_step": wl.elements * esz, "d2h_bytes_per_step": wl.elements * esz,
            "ms_per_step": round(ms, 4), "steps": steps,
            "pipeline": f"{ngroups} launches of about equal size, upload / step / read-back "
                        "on three streams, device gradient double-buffered"}


def run_codec(args, wl):
    """The stand-alone block-wise quantize or dequantize of one tensor, timed
    like a step (L2 flushed before each, CUDA events on the stream)."""
    import torch
    import bit_block_wise_gb300 as bnb8
    from bit_block_wise_gb300 import build as bnb8_build

    world, rank, local = setup_dist()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    bnb8_build.build()
    stream = torch.cuda.current_stream()
    n, B = wl.elements, wl.blocksize
    nb = -(-n // B)
    q = bnb8.bnb8_create_qmap(True).to(device)
    x = workloads.torch_normal_with_outliers(n, wl.grad[1], wl.grad[2], wl.grad[3], 11 + rank,
                                             device, torch.float32)
    codes = torch.empty(n, dtype=torch.uint8, device=device)
    absmax = torch.empty(nb, dtype=torch.float32, device=device)
    out = torch.empty(n, dtype=torch.float32, device=device)
    bnb8.bnb8_quantize_blockwise(x, q, B, codes, absmax, stream=stream)
    quant = wl.op == "quantize"

    def one_step():
        if quant:
            bnb8.bnb8_quantize_blockwise(x, q, B, codes, absmax, stream=stream)
        else:
            bnb8.bnb8_dequantize_blockwise(codes, absmax, q, B, out=out, stream=stream)

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    flush_read = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)
    flush_sink = torch.empty((), dtype=torch.int32, device=device)
    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    sampler = ClockSampler() if rank == 0 else None
    time.sleep(0.3 if sampler else 0.0)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    for k in range(args.steps):
        if k % HOST_AHEAD_STEPS == 0:
            gpu_sleep(stream, HOST_AHEAD_STEPS * HOST_AHEAD_US_PER_STEP)
        flush.zero_()
        torch.amax(flush_read, 0, out=flush_sink)
        starts[k].record(stream)
        one_step()
        ends[k].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    rows = sampler.stop() if sampler else []
    dist_ms = step_distribution([s.elapsed_time(e) for s, e in zip(starts, ends)])
    ms = max_over_ranks(dist_ms["median"], world, device)

    # end to end: the input from pinned host memory, the output read back
    steps_e2e = max(3, min(args.steps, 50))
    if quant:
        h_in = torch.empty(n, dtype=torch.float32, pin_memory=True)
        h_in.copy_(x)
        h_codes = torch.empty(n, dtype=torch.uint8, pin_memory=True)
        h_absmax = torch.empty(nb, dtype=torch.float32, pin_memory=True)
    else:
        h_codes = torch.empty(n, dtype=torch.uint8, pin_memory=True)
        h_codes.copy_(codes)
        h_absmax = torch.empty(nb, dtype=torch.float32, pin_memory=True)
        h_absmax.copy_(absmax)
        h_out = torch.empty(n, dtype=torch.float32, pin_memory=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps_e2e):
        if quant:
            x.copy_(h_in, non_blocking=True)
            one_step()
            h_codes.copy_(codes, non_blocking=True)
            h_absmax.copy_(absmax, non_blocking=True)
        else:
            codes.copy_(h_codes, non_blocking=True)
            absmax.copy_(h_absmax, non_blocking=True)
            one_step()
            h_out.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = e0.elapsed_time(e1) / steps_e2e
    in_b, out_b = (n * 4, n + nb * 4) if quant else (n + nb * 4, n * 4)

    alg = wl.algorithmic_bytes()
    peak, peak_kind = hbm_peak()
    achieved = alg / (ms * 1e-3) / 1e9
    res = {
        "metric": METRIC, "value": round(world * n / (ms * 1e-3) / 1e9, 3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 5), "step_ms": {k: round(v, 5) for k, v in dist_ms.items()},
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.desc, "name": wl.name, "elements": n, "blocksize": B,
                   "l2": "flushed before every timed step (256 MiB written, then 256 MiB of "
                         "other data read, leaving clean unrelated lines)",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                     "algorithmic_bytes_per_step": alg, "traffic": ncu_traffic(wl.name)},
        "e2e": {"value": round(n / (ms_e2e * 1e-3) / 1e9, 3), "unit": UNIT,
                "h2d_bytes_per_step": in_b, "d2h_bytes_per_step": out_b,
                "ms_per_step": round(ms_e2e, 4), "steps": steps_e2e,
                "pipeline": "upload, convert and read back in stream order"},
        "gpu_launches": args.steps,
        "clocks": summarize_clocks(rows, t0, t1),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = codec_baseline(wl, args.cpu_budget)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def codec_baseline(wl, budget_s):
    """The oracle's quantize / dequantize on a bounded leading sample."""
    import oracle
    oracle.build()
    B = wl.blocksize
    q = oracle.create_qmap(True)
    n = min(wl.elements, 64 * B)
    done_n, t0 = 0, time.perf_counter()
    while True:
        x = workloads.normal_with_outliers(n, wl.grad[1], wl.grad[2], wl.grad[3], 3)
        if wl.op == "quantize":
            t1 = time.perf_counter()
            oracle.quantize_blockwise(x, "f32", q, B)
        else:
            c, a = oracle.quantize_blockwise(x, "f32", q, B)
            t1 = time.perf_counter()
            oracle.dequantize_blockwise(c, a, q, B, "f32")
        el = time.perf_counter() - t1
        done_n += n
        if time.perf_counter() - t0 > budget_s / 2 or n >= wl.elements:
            break
        n = int(min(wl.elements, max(n, n * min(8.0, budget_s / 4 / max(el, 1e-6)))))
        n -= n % B
    value = n / el / 1e9
    return {"value": round(value, 6), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n:,} of the workload's {wl.elements:,} elements, one {wl.op}, "
                      f"single-threaded C oracle, {el:.2f} s"}


# ---------------------------------------------------------------------------
# the CPU oracle (baseline leg and --impl reference)
# ---------------------------------------------------------------------------
def _gran(wl):
    """Sample granularity (elements) of the oracle legs: the block size, or
    256 for tensor-wise quantization (where the sample is one block)."""
    return wl.blocksize or 256


def _oracle_b(wl, n):
    """The oracle's block size for a sample of n elements."""
    return wl.blocksize or n


def _oracle_sample(wl, n_sample, params=None):
    """Host copies of the first n_sample elements of the workload's first
    tensor (device state when given, else fresh seeded values)."""
    import oracle
    n = min(n_sample, wl.sizes[0])
    B = _oracle_b(wl, n)
    dt = wl.dtype
    p = oracle.to_storage(workloads.normal(n, wl.p_std, 1), dt)
    q1 = oracle.create_qmap(wl.optim not in ("rmsprop", "adagrad"))
    q2 = oracle.create_qmap(False)
    st = oracle.zero_state(wl.optim, n, 8, B, q1, q2)
    t = oracle.TensorState(p, *st, 8)
    if wl.grad[0] == "outliers":
        g = workloads.normal_with_outliers(n, wl.grad[1], wl.grad[2], wl.grad[3], 2)
    elif wl.grad[0] == "rows":
        cols = wl.grad[2]
        g = workloads.sparse_rows(max(1, n // cols), cols, wl.grad[3], wl.grad[4], 2)[:n]
        if g.size < n:
            g = np.concatenate([g, np.zeros(n - g.size, np.float32)])
    else:
        g = workloads.normal(n, wl.grad[1], 2)
    return t, oracle.to_storage(g, dt), q1, q2


def time_oracle(wl, n_sample, steps, budget_s):
    import oracle
    oracle.build()
    t, g, q1, q2 = _oracle_sample(wl, n_sample)
    hp_kw = {k: v for k, v in wl.hp.items()}
    done = 0
    t0 = time.perf_counter()
    for k in range(1, steps + 1):
        oracle.step(oracle.HParams(optim=wl.optim, step=k, **hp_kw), t, g, wl.dtype,
                    _oracle_b(wl, t.p.size), q1, q2)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    el = time.perf_counter() - t0
    return t.p.size, done, el


def calibrate_oracle(wl):
    n, done, el = time_oracle(wl, 16 * _gran(wl), 2, 10.0)
    return el / done / n  # seconds per element


def _host_bits(t):
    """A device tensor as numpy: float32 as float32, 16-bit floats as their
    uint16 patterns (the oracle's storage form), others as they are."""
    import torch
    t = t.detach().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def sampled_parity(wl, params, gpu_step, step, grads, nsample=48, seed=7):
    """The oracle's check of one GPU step on sampled blocks of the first 8-bit
    tensor: the blocks' p, g, codes and absmax are copied out, the GPU steps
    the whole workload once, and the oracle steps the copies.  Reports the
    share of code mismatches and their largest index distance (the method
    allows at most one index, at exact ties), plus absmax and p mismatches
    (p only where no max_unorm multiplier enters: the per-tensor one needs
    the whole tensor, and either matches its definition to 1e-6, not bit
    for bit)."""
    import torch
    import oracle
    oracle.build()
    idx = next((i for i, ps in enumerate(params) if ps.state_bits == 8), None)
    B = wl.blocksize
    if idx is None or B == 0:
        return None
    ps = params[idx]
    n = ps.p.numel()
    nb = -(-n // B)
    rng = np.random.default_rng(seed)
    blocks = sorted(set(rng.choice(nb, size=min(nsample, nb), replace=False).tolist()) | {0, nb - 1})
    full = [b for b in blocks if (b + 1) * B <= n]
    part = [b for b in blocks if (b + 1) * B > n]
    two = ps.s1.numel() == 2 * n  # AdEMAMix: m1 and m2 stacked

    def elems(group, base=0):
        return torch.cat([torch.arange(base + b * B, base + min(n, (b + 1) * B), device=ps.p.device)
                          for b in group])

    def snapshot(group):
        e = elems(group)
        bi = torch.tensor(group, device=ps.p.device)
        s1 = torch.cat([ps.s1[e], ps.s1[elems(group, n)]]) if two else ps.s1[e]
        a1 = torch.cat([ps.absmax1[bi], ps.absmax1[bi + nb]]) if two else ps.absmax1[bi]
        return oracle.TensorState(_host_bits(ps.p[e]), _host_bits(s1),
                                  None if ps.s2 is None else _host_bits(ps.s2[e]), _host_bits(a1),
                                  None if ps.absmax2 is None else _host_bits(ps.absmax2[bi]), 8)

    before = [(g, snapshot(g), _host_bits(grads[idx][elems(g)])) for g in (full, part) if g]
    gpu_step()
    if ps.p.is_cuda:
        torch.cuda.synchronize()
    q1 = oracle.create_qmap(wl.optim not in ("rmsprop", "adagrad"))
    q2 = oracle.create_qmap(False)
    hp = oracle.HParams(optim=wl.optim, step=step, **wl.hp)
    # p bit for bit only where no max_unorm multiplier enters (the per-tensor
    # one needs the whole tensor; both match the definition to 1e-6)
    compare_p = not wl.hp.get("max_unorm", 0.0) > 0
    codes = mism = maxd = am_bad = p_bad = p_total = 0
    for group, ref, g in before:
        got = snapshot(group)
        oracle.step(hp, ref, g, wl.dtype, B, q1, q2)
        for a, b in ((got.s1, ref.s1), (got.s2, ref.s2)):
            if a is None:
                continue
            d = np.abs(a.astype(np.int32) - b.astype(np.int32))
            codes += d.size
            mism += int(np.count_nonzero(d))
            maxd = max(maxd, int(d.max()) if d.size else 0)
        for a, b in ((got.absmax1, ref.absmax1), (got.absmax2, ref.absmax2)):
            if a is not None:
                am_bad += int(np.count_nonzero(a.view(np.uint32) != b.view(np.uint32)))
        if compare_p:
            p_total += got.p.size
            if got.p.size:
                differ = (got.p.view(np.uint8).reshape(got.p.size, -1) !=
                          ref.p.view(np.uint8).reshape(ref.p.size, -1))
                p_bad += int(differ.any(axis=1).sum())
    return {"kind": "oracle", "blocks": len(blocks), "codes": codes,
            "code_mismatch_rate": mism / max(codes, 1), "code_mismatches": mism,
            "code_mismatch_max_index_delta": maxd, "absmax_mismatches": am_bad,
            "p_compared": p_total, "p_mismatches": p_bad if compare_p else None,
            "step": step, "tensor": idx}


def cpu_baseline(wl, params=None, budget_s=15.0):
    sec_per_elem = calibrate_oracle(wl)
    G = _gran(wl)
    n_sample = int(max(G, min(wl.sizes[0], budget_s / 3 / sec_per_elem)))
    n_sample -= n_sample % G or 0
    n_sample = max(G, n_sample)
    n, done, el = time_oracle(wl, n_sample, 3, budget_s)
    value = n * done / el / 1e9
    return {"value": round(value, 6), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n:,} of the workload's {wl.elements:,} elements (first tensor, "
                      f"{'tensor-wise' if not wl.blocksize else f'{n // wl.blocksize:,} blocks'}), "
                      f"{done} step(s), single-threaded C oracle, "
                      f"{el:.1f} s"}


def run_reference(args, wl):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    if wl.op != "step":
        base = codec_baseline(wl, args.ref_budget)
        print(json.dumps({"impl": "reference", "metric": METRIC, "value": base["value"],
                          "unit": UNIT, "n_gpus": world, "steps": args.steps,
                          "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
                          "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
                          "config": {"workload": wl.desc, "name": wl.name,
                                     "elements": wl.elements, "blocksize": wl.blocksize},
                          "cpu_baseline": base,
                          "e2e": {"value": base["value"], "unit": UNIT, "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return
    total_budget = args.ref_budget
    sec_per_elem = calibrate_oracle(wl)
    per_step = total_budget / max(1, args.steps + args.warmup)
    G = _gran(wl)
    n_sample = int(max(G, min(wl.sizes[0], per_step / sec_per_elem)))
    n_sample = max(G, n_sample - n_sample % G)
    import oracle
    t, g, q1, q2 = _oracle_sample(wl, n_sample)
    for k in range(1, args.warmup + 1):
        oracle.step(oracle.HParams(optim=wl.optim, step=k, **wl.hp), t, g, wl.dtype,
                    _oracle_b(wl, t.p.size), q1, q2)
    t0 = time.perf_counter()
    for k in range(args.warmup + 1, args.warmup + args.steps + 1):
        oracle.step(oracle.HParams(optim=wl.optim, step=k, **wl.hp), t, g, wl.dtype,
                    _oracle_b(wl, t.p.size), q1, q2)
    el = time.perf_counter() - t0
    n = t.p.size
    value = n * args.steps / el / 1e9
    sample = (f"{n:,} of the workload's {wl.elements:,} elements per step "
              f"({n // _gran(wl):,} blocks of {_gran(wl)} of the first tensor"
              f"{', tensor-wise' if not wl.blocksize else ''}), single-threaded C oracle")
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
           "config": {"workload": wl.desc, "name": wl.name, "elements": wl.elements,
                      "blocksize": wl.blocksize, "optimizer": wl.optim},
           "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": 1, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--l2", default="flush", choices=["flush", "none", "auto"],
                    help="between timed steps: flush the L2, or run back to back when the "
                         "step's inputs exceed the L2 (none, auto: back to back where allowed)")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle time for the cpu_baseline leg")
    ap.add_argument("--ref-budget", type=float, default=90.0,
                    help="seconds of oracle time for --impl reference (all steps)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    wl = WORKLOADS[args.workload]()
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_gpu(args, wl)


if __name__ == "__main__":
    main()
