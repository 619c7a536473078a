"""torch.optim-style optimizers over the library's 8-bit block-wise step.

The classes follow the parameter lists of the bitsandbytes docs page
"optim_overview.md" (Optimizer8bit / Optimizer2State / Optimizer1State:
lr, betas, eps, weight_decay, optim_bits, min_8bit_size, max_unorm,
skip_zeros, alpha, t_alpha, t_beta3) and its GlobalOptimManager (per-parameter
overrides of any of them, e.g. 32-bit state for one weight).  Everything a
step computes runs in the library's kernels; this module only keeps the
per-parameter state and batches parameters into library calls.

Differences from that page, stated: optim_bits defaults to 8 (the classes here
exist for the 8-bit path); blocksize (256) and the per-block max_unorm reading
(unorm_per_block) are exposed.

Paged optimizers (is_paged=True, and the Paged* classes that the benchmark
script of "[XPU] Implemented 8bit optimizers in triton #1692" lists): every
state array lives in paged (CUDA managed) memory, which the driver moves to
the host when the device runs short.  The states that one step creates share
one paged buffer, and each step first prefetches the buffers of the
parameters it updates to their device, on the step's stream: one call per
buffer, whose pages the step then finds resident instead of faulting them in
(several times slower).  page_prefetch=False leaves placement to the driver:
no per-step call, which saves its cost when the states stay resident.

carry_pnorm=True (with max_unorm per tensor): each batch keeps its workspace
from step to step, and the library carries ||p|| from one step to the next
(hparams flag BNB8_CARRY_PNORM) instead of reading p again for it.  The
parameters must then change only through this optimizer between steps;
load_state_dict() and invalidate_carried_norms() drop the carried norms.
"""
from __future__ import annotations

import torch

from . import HParams, ParamState, bnb8_create_qmap, bnb8_workspace_size, paged_prefetch, \
    paged_zero_states, step as _step, zero_state

_HPARAM_KEYS = ("lr", "betas", "eps", "weight_decay", "optim_bits", "min_8bit_size", "max_unorm",
                "skip_zeros", "alpha", "t_alpha", "t_beta3", "blocksize", "unorm_per_block")


class OptimManager:
    """Per-parameter overrides of the optimizer config (the docs'
    GlobalOptimManager).  Parameters are identified by object, which survives
    ``model.cuda()`` (it moves a Parameter's data in place), so registering
    them first is optional."""

    _instance = None

    def __init__(self):
        self._overrides = {}

    @classmethod
    def get_instance(cls) -> "OptimManager":
        if cls._instance is None:
            cls._instance = cls()
        return cls._instance

    def register_parameters(self, params):
        for p in params if not isinstance(params, torch.Tensor) else [params]:
            self._overrides.setdefault(id(p), {})

    def override_config(self, parameters, key=None, value=None, key_value_dict=None):
        kv = dict(key_value_dict or {})
        if key is not None:
            kv[key] = value
        for k in kv:
            if k not in _HPARAM_KEYS:
                raise ValueError(f"unknown optimizer setting {k!r}")
        params = [parameters] if isinstance(parameters, torch.Tensor) else list(parameters)
        for p in params:
            self._overrides.setdefault(id(p), {}).update(kv)

    def config_of(self, p) -> dict:
        return self._overrides.get(id(p), {})

    def clear(self):
        self._overrides.clear()


class Optimizer8bit(torch.optim.Optimizer):
    """One optimizer of the library (``optim`` = adam, adamw, momentum,
    rmsprop, adagrad, lion, ademamix) with 8-bit block-wise states.

    Tensors with fewer than ``min_8bit_size`` elements, or configured with
    ``optim_bits=32``, keep 32-bit states.  Each ``step()`` makes one library
    call per batch of parameters that share a dtype, a config and an update
    number (usually one call per parameter group).  Gradients must be dense
    and of the parameter's dtype; parameters must be contiguous."""

    def __init__(self, params, optim="adam", lr=1e-3, betas=(0.9, 0.999), eps=1e-8,
                 weight_decay=0.0, optim_bits=8, min_8bit_size=4096, max_unorm=0.0,
                 skip_zeros=False, alpha=0.0, t_alpha=0, t_beta3=0, blocksize=256,
                 unorm_per_block=False, is_paged=False, page_prefetch=True,
                 carry_pnorm=False, manager: OptimManager | None = None):
        if optim not in ("adam", "adamw", "momentum", "rmsprop", "adagrad", "lion", "ademamix"):
            raise ValueError(f"unknown optimizer {optim!r}")
        if optim_bits not in (8, 32):
            raise ValueError("optim_bits must be 8 or 32")
        defaults = dict(lr=lr, betas=tuple(betas), eps=eps, weight_decay=weight_decay,
                        optim_bits=optim_bits, min_8bit_size=min_8bit_size, max_unorm=max_unorm,
                        skip_zeros=skip_zeros, alpha=alpha, t_alpha=t_alpha or 0,
                        t_beta3=t_beta3 or 0, blocksize=blocksize,
                        unorm_per_block=unorm_per_block)
        super().__init__(params, defaults)
        self.optim = optim
        self.is_paged = bool(is_paged)
        self.page_prefetch = bool(page_prefetch)
        self.carry_pnorm = bool(carry_pnorm)
        self.manager = manager or OptimManager.get_instance()
        self._maps = {}
        self._carry_ws = {}  # batch -> workspace kept between steps (carry_pnorm)

    # ---- configuration ------------------------------------------------------
    def _config(self, group, p) -> dict:
        cfg = {k: group[k] for k in _HPARAM_KEYS}
        cfg.update(self.manager.config_of(p))
        return cfg

    def _maps_for(self, device):
        key = str(device)
        if key not in self._maps:
            s = bnb8_create_qmap(True).to(device)
            u = bnb8_create_qmap(False).to(device)
            # RMSprop and Adagrad keep a non-negative single state
            self._maps[key] = (u, None) if self.optim in ("rmsprop", "adagrad") else \
                (s, u if self.optim in ("adam", "adamw", "ademamix") else None)
        return self._maps[key]

    @staticmethod
    def _bits(p, cfg) -> int:
        return 8 if cfg["optim_bits"] == 8 and p.numel() >= cfg["min_8bit_size"] else 32

    @staticmethod
    def _state_dict_of(bits, arrays) -> dict:
        st = {"step": 0, "state_bits": bits}
        for key, a in zip(("state1", "state2", "absmax1", "absmax2"), arrays):
            if a is not None:
                st[key] = a
        return st

    def _init_states(self, todo, bits_of=None) -> None:
        """Zero states (codes of 0.0, absmax 0, or binary32 zeros) of the
        (p, cfg) pairs in todo, on each p's device, with the state bits of
        bits_of[p] if given, else of cfg; paged: one paged buffer per device
        for all of them."""
        bits = {p: (bits_of or {}).get(p) or self._bits(p, cfg) for p, cfg in todo}
        if not self.is_paged:
            for p, cfg in todo:
                self.state[p].update(self._state_dict_of(
                    bits[p], zero_state(p.data, self.optim, bits[p], cfg["blocksize"])))
            return
        by_dev = {}
        for p, cfg in todo:
            by_dev.setdefault(p.device, []).append((p, cfg))
        for items in by_dev.values():
            specs = [(p.data, self.optim, bits[p], cfg["blocksize"]) for p, cfg in items]
            for (p, _), arrays in zip(items, paged_zero_states(specs)):
                self.state[p].update(self._state_dict_of(bits[p], arrays))

    # ---- the update ---------------------------------------------------------
    @torch.no_grad()
    def step(self, closure=None):
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        batches = {}
        live, todo = [], []
        for gi, group in enumerate(self.param_groups):
            for p in group["params"]:
                if p.grad is None:
                    continue
                if p.grad.is_sparse:
                    raise RuntimeError("sparse gradients are not supported")
                if not p.is_contiguous() or not p.grad.is_contiguous():
                    raise RuntimeError("parameters and gradients must be contiguous")
                if p.grad.dtype != p.dtype:
                    raise RuntimeError("the gradient must have the parameter's dtype")
                cfg = self._config(group, p)
                live.append((gi, p, cfg))
                if len(self.state[p]) == 0:
                    todo.append((p, cfg))
        self._init_states(todo)
        for gi, p, cfg in live:
            st = self.state[p]
            st["step"] += 1
            key = (gi, str(p.device), p.dtype, st["step"],
                   tuple((k, cfg[k]) for k in _HPARAM_KEYS if k not in ("optim_bits", "min_8bit_size")))
            batches.setdefault(key, (cfg, []))[1].append(p)
        for (gi, dev, dtype, k, _), (cfg, params) in batches.items():
            b1, b2 = cfg["betas"][0], cfg["betas"][1]
            b3 = cfg["betas"][2] if len(cfg["betas"]) > 2 else 0.9999
            hp = HParams(optim=self.optim, lr=cfg["lr"], beta1=b1, beta2=b2, beta3=b3,
                         alpha=cfg["alpha"], eps=cfg["eps"], weight_decay=cfg["weight_decay"],
                         max_unorm=cfg["max_unorm"], step=k, t_alpha=cfg["t_alpha"],
                         t_beta3=cfg["t_beta3"], skip_zeros=cfg["skip_zeros"],
                         blocksize=cfg["blocksize"], unorm_per_block=cfg["unorm_per_block"])
            states = []
            stream = torch.cuda.current_stream(params[0].device)
            if self.is_paged and self.page_prefetch:
                # each paged buffer once (the batch's states usually share one)
                paged_prefetch([self.state[p].get(key) for p in params
                                for key in ("state1", "state2", "absmax1", "absmax2")],
                               params[0].device, stream)
            for p in params:
                st = self.state[p]
                states.append(ParamState(p.data, p.grad, st["state1"], st.get("state2"),
                                         st.get("absmax1"), st.get("absmax2"), st["state_bits"]))
            q1, q2 = self._maps_for(params[0].device)
            ws = None
            if (self.carry_pnorm and hp.max_unorm > 0 and not hp.unorm_per_block and
                    hp.blocksize != 0 and not hp.skip_zeros):
                hp.carry_pnorm = True
                ws = self._carry_workspace((gi, dev, dtype, tuple(p.data_ptr() for p in params)),
                                           states, hp)
            _step(states, hp, q1, q2, workspace=ws, stream=stream)
        return loss

    def _carry_workspace(self, key, states, hp):
        need = bnb8_workspace_size(states, hp)
        ws = self._carry_ws.get(key)
        if ws is None or ws.numel() < need:
            ws = torch.zeros(need, dtype=torch.uint8, device=states[0].p.device)
            self._carry_ws[key] = ws
        return ws

    def invalidate_carried_norms(self):
        """Forget the carried ||p|| of every batch: call after changing
        parameters outside step() when carry_pnorm is on."""
        self._carry_ws.clear()

    # ---- checkpoints --------------------------------------------------------
    def load_state_dict(self, state_dict):
        """torch's loader casts every state tensor of a floating-point
        parameter to the parameter's dtype (uint8 codes included); here every
        state tensor keeps the dtype it was saved with, bit for bit."""
        saved = state_dict["state"]
        self.invalidate_carried_norms()
        super().load_state_dict(state_dict)
        params = [(g, p) for g in self.param_groups for p in g["params"]]
        if self.is_paged:
            # the restored states of each device share one paged buffer again
            todo = [(params[idx][1], self._config(*params[idx])) for idx in saved
                    if params[idx][1].is_cuda]
            self._init_states(todo, {params[idx][1]: st.get("state_bits")
                                     for idx, st in saved.items()})
        for idx, st in saved.items():
            p = params[idx][1]
            for key, val in st.items():
                if not torch.is_tensor(val):
                    continue
                mine = self.state[p].get(key) if self.is_paged and p.is_cuda else None
                if mine is not None and mine.shape == val.shape and mine.dtype == val.dtype:
                    mine.copy_(val)
                else:
                    self.state[p][key] = val.to(device=p.device)
            for key in ("step", "state_bits"):
                if key in st:
                    self.state[p][key] = st[key]


def _named(optim, doc_defaults):
    def init(self, params, **kw):
        args = dict(doc_defaults)
        args.update(kw)
        Optimizer8bit.__init__(self, params, optim=optim, **args)
    return init


class Adam8bit(Optimizer8bit):
    """Adam with 8-bit block-wise states (decay coupled into g, as torch.optim.Adam)."""
    __init__ = _named("adam", {})


class AdamW8bit(Optimizer8bit):
    """AdamW with 8-bit block-wise states (decoupled decay, default 1e-2)."""
    __init__ = _named("adamw", {"weight_decay": 1e-2})


class Momentum8bit(Optimizer8bit):
    """SGD with momentum (beta1) and 8-bit block-wise state."""
    __init__ = _named("momentum", {"lr": 1e-2, "betas": (0.9, 0.0)})


class RMSprop8bit(Optimizer8bit):
    """RMSprop (beta1 = alpha of torch.optim.RMSprop) with 8-bit state."""
    __init__ = _named("rmsprop", {"lr": 1e-2, "betas": (0.99, 0.0)})


class Adagrad8bit(Optimizer8bit):
    """Adagrad with 8-bit state."""
    __init__ = _named("adagrad", {"lr": 1e-2, "betas": (0.0, 0.0), "eps": 1e-10})


class Lion8bit(Optimizer8bit):
    """Lion with 8-bit state."""
    __init__ = _named("lion", {"lr": 1e-4, "betas": (0.9, 0.99)})


class AdEMAMix8bit(Optimizer8bit):
    """AdEMAMix with 8-bit states (betas = (beta1, beta2, beta3))."""
    __init__ = _named("ademamix", {"betas": (0.9, 0.999, 0.9999), "alpha": 5.0,
                                   "weight_decay": 1e-2})


class PagedAdam8bit(Optimizer8bit):
    """Adam8bit with paged states."""
    __init__ = _named("adam", {"is_paged": True})


class PagedAdamW8bit(Optimizer8bit):
    """AdamW8bit with paged states."""
    __init__ = _named("adamw", {"weight_decay": 1e-2, "is_paged": True})


class PagedLion8bit(Optimizer8bit):
    """Lion8bit with paged states."""
    __init__ = _named("lion", {"lr": 1e-4, "betas": (0.9, 0.99), "is_paged": True})


class PagedAdEMAMix8bit(Optimizer8bit):
    """AdEMAMix8bit with paged states."""
    __init__ = _named("ademamix", {"betas": (0.9, 0.999, 0.9999), "alpha": 5.0,
                                   "weight_decay": 1e-2, "is_paged": True})
