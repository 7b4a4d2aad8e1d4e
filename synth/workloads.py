"""Synthetic workloads: tensor shapes, dtypes, seeds and input scales.

Inputs only; no optimizer arithmetic. Shared by the tests (oracle side and
GPU side) and the benchmark so both run on the same seeded data.

Shapes follow the five benchmark configurations the optimizer is measured
on. Where the description leaves a value open, the reading used is stated
here:
  * parameter init std 0.02 where unstated;
  * Muon lr 0.02, wd 0.01, momentum 0.95 (Nesterov) in every configuration;
  * AdamW lr 3e-4 (the Speedtronic "Configuration" example), betas 0.9/0.95,
    eps 1e-8, wd 0.1 on every AdamW tensor;
  * "N(0,1e-3)" means std 1e-3; "lognormal(0,1) per tensor" is one factor
    exp(z) per tensor, z drawn from the generator.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import lognormal_factor

SEED = 0

KIND_W, KIND_G, KIND_AW, KIND_AG = 0, 1, 2, 3


def tensor_id(kind: int, index: int, step: int = 0) -> int:
    """Generator stream of (kind, tensor index, step)."""
    return (index << 24) | (kind << 16) | step


@dataclass
class MuonSpec:
    name: str
    views: int
    rows: int
    cols: int
    param_dtype: str = "bf16"
    grad_dtype: str = "bf16"
    w_std: float = 0.02
    g_std: float = 1e-3
    lognormal: bool = False
    lr_mult: float = 1.0
    wd: float = 0.01

    @property
    def numel(self) -> int:
        return self.views * self.rows * self.cols

    @property
    def shape(self):
        return (self.views * self.rows, self.cols)


@dataclass
class AdamSpec:
    name: str
    shape: tuple
    param_dtype: str = "bf16"
    grad_dtype: str = "bf16"
    w_std: float = 0.02
    g_std: float = 1e-3
    lognormal: bool = False
    lr_mult: float = 1.0
    wd: float = 0.1
    w_const: float | None = None  # norms start at a constant (1.0)

    @property
    def numel(self) -> int:
        return int(np.prod(self.shape))


@dataclass
class Workload:
    name: str
    muon: list = field(default_factory=list)
    adamw: list = field(default_factory=list)
    muon_hp: dict = field(default_factory=dict)
    adam_hp: dict = field(default_factory=dict)
    steps: int = 1
    seed: int = SEED
    state_dtype: str = "f32"   # optimizer state: "f32", or "bf16" kept stochastically rounded
    param_sr: bool = False     # bf16 parameters written stochastically rounded

    def grad_std(self, kind: int, index: int) -> np.float32:
        spec = (self.muon if kind == KIND_G else self.adamw)[index]
        std = np.float32(spec.g_std)
        if spec.lognormal:
            std = np.float32(std * lognormal_factor(self.seed, tensor_id(kind, index)))
        return std

    @property
    def muon_elems(self) -> int:
        return sum(s.numel for s in self.muon)

    @property
    def adam_elems(self) -> int:
        return sum(s.numel for s in self.adamw)


MUON_HP = dict(lr=0.02, momentum=0.95, nesterov=True, eps=1e-7, ns_steps=5,
               coeffs=(3.4445, -4.7750, 2.0315))
ADAM_HP = dict(lr=3e-4, betas=(0.9, 0.95), eps=1e-8)


def single_matrix() -> Workload:
    """256 x 1024 fp32, W and G ~ N(0, 1), zero momentum, one step."""
    return Workload(
        name="single_256x1024_fp32",
        muon=[MuonSpec("W", 1, 256, 1024, "f32", "f32", w_std=1.0, g_std=1.0)],
        muon_hp=dict(MUON_HP), adam_hp=dict(ADAM_HP), steps=1)


def gpt124m() -> Workload:
    """d=768, 12 layers: Q/K/V/O 768^2, gate_up (2, 2048, 768), down 768 x 2048
    on Muon; embedding 50304 x 768 and two RMSNorm vectors per layer on
    AdamW. bf16 params and grads, grads N(0,1e-3) * lognormal per tensor."""
    muon, adamw = [], []
    for l in range(12):
        for nm in ("q", "k", "v", "o"):
            muon.append(MuonSpec(f"l{l}.{nm}", 1, 768, 768, lognormal=True))
        muon.append(MuonSpec(f"l{l}.gate_up", 2, 2048, 768, lognormal=True))
        muon.append(MuonSpec(f"l{l}.down", 1, 768, 2048, lognormal=True))
    adamw.append(AdamSpec("embed", (50304, 768), lognormal=True))
    for l in range(12):
        for k in range(2):
            adamw.append(AdamSpec(f"l{l}.norm{k}", (768,), lognormal=True, w_const=1.0))
    return Workload("gpt124m_d768_l12", muon, adamw, dict(MUON_HP), dict(ADAM_HP), steps=10)


def llama7b(layers: int = 32, vocab_rows: int = 128256) -> Workload:
    """d=4096, 32 layers, GQA: Q/O 4096^2, K/V 1024 x 4096, gate_up
    (2, 14336, 4096), down 4096 x 14336 on Muon; untied embedding and head
    128256 x 4096 plus 65 norms on AdamW; bf16 params/grads, fp32 state.
    ``layers`` / ``vocab_rows`` give a slice of the same shapes (profiling)."""
    muon, adamw = [], []
    for l in range(layers):
        muon.append(MuonSpec(f"l{l}.q", 1, 4096, 4096))
        muon.append(MuonSpec(f"l{l}.k", 1, 1024, 4096))
        muon.append(MuonSpec(f"l{l}.v", 1, 1024, 4096))
        muon.append(MuonSpec(f"l{l}.o", 1, 4096, 4096))
        muon.append(MuonSpec(f"l{l}.gate_up", 2, 14336, 4096))
        muon.append(MuonSpec(f"l{l}.down", 1, 4096, 14336))
    adamw.append(AdamSpec("embed", (vocab_rows, 4096)))
    adamw.append(AdamSpec("head", (vocab_rows, 4096)))
    for k in range(2 * layers + 1):
        adamw.append(AdamSpec(f"norm{k}", (4096,), w_const=1.0))
    name = ("llama7b_d4096_l32" if (layers, vocab_rows) == (32, 128256)
            else f"llama7b_slice_l{layers}_v{vocab_rows}")
    return Workload(name, muon, adamw, dict(MUON_HP), dict(ADAM_HP), steps=1)


def llama7b_layer() -> Workload:
    """One layer of the 7B-shape set (every Newton-Schulz shape class, 7 views)
    with an 8192-row slice of embedding and head: about 3.5 GB on the device,
    small enough for a multi-pass profile of every kernel of the step."""
    return llama7b(layers=1, vocab_rows=8192)


def llama7b_bf16_state() -> Workload:
    """The 7B-shape set with bf16 optimizer state (Muon momentum, Adam
    moments) and bf16 parameters, all written stochastically rounded
    (dew.training.optim "bf16_moments", "stochastic_round_bf16")."""
    wl = llama7b()
    wl.name = "llama7b_d4096_l32_bf16state"
    wl.state_dtype = "bf16"
    wl.param_sr = True
    return wl


def gpt124m_bf16_state() -> Workload:
    """The 124M set with bf16 optimizer state and stochastically rounded
    bf16 parameters (a small case of the bf16-state path)."""
    wl = gpt124m()
    wl.name = "gpt124m_d768_l12_bf16state"
    wl.state_dtype = "bf16"
    wl.param_sr = True
    return wl


def moe_mla(experts: int = 64) -> Workload:
    """One MoE layer with 64 experts (gate_up (2, 1408, 2048) as two wide
    views, down 2048 x 1408 tall) and the MLA kv up-projection, 32 heads x
    (128 K + 128 V rows) x 512, as 64 views of 128 x 512. NorMuon (beta2 0.95),
    Muon+ row_col and cautious weight decay on."""
    muon = []
    for e in range(experts):
        muon.append(MuonSpec(f"e{e}.gate_up", 2, 1408, 2048))
        muon.append(MuonSpec(f"e{e}.down", 1, 2048, 1408))
    muon.append(MuonSpec("mla.kv_b", 64, 128, 512))
    hp = dict(MUON_HP, normuon=True, beta2=0.95, muon_plus=True, cautious=1)
    return Workload(f"moe{experts}_mla_all_variants", muon, [], hp, dict(ADAM_HP), steps=1)


def moe_mla_e16() -> Workload:
    """The same layer with 16 experts (about 1.2 GB of parameters, gradients
    and momentum): a profiler-sized case of the same passes."""
    return moe_mla(16)


def moe_mla_e16_cu() -> Workload:
    """The 16-expert layer with the cautious-update mask (Speedtronic
    "Cautious updates") in place of the cautious weight decay: the apply pass
    then reads the gradient too."""
    wl = moe_mla(16)
    wl.name = "moe16_mla_cautious_update"
    wl.muon_hp = dict(wl.muon_hp, cautious=2)
    return wl


def ns_sweep_shapes(max_x_bytes: int = 64 * 2 ** 30):
    """Newton-Schulz-only sweep: square n x n, wide n x 4n and tall 4n x n for
    n in {512 .. 8192}, batch counts 1..256 capped at `max_x_bytes` of bf16
    operand X (64 GiB by default)."""
    out = []
    for n in (512, 1024, 2048, 4096, 8192):
        for aspect, (r, c) in (("1:1", (n, n)), ("1:4", (n, 4 * n)), ("4:1", (4 * n, n))):
            for batch in (1, 4, 16, 64, 256):
                if batch * r * c * 2 > max_x_bytes:
                    continue
                out.append((aspect, n, batch, r, c))
    return out


def adamw_2p30(log2_elems: int = 30) -> Workload:
    """AdamW alone on 2^30 fp32 elements (HBM roofline case)."""
    return Workload(f"adamw_2p{log2_elems}_fp32",
                    [], [AdamSpec("flat", (1 << log2_elems,), "f32", "f32", w_std=1.0, g_std=1e-3)],
                    dict(MUON_HP), dict(ADAM_HP), steps=1)


def adamw_2p26() -> Workload:
    """The same on 2^26 elements (1.8 GB on the device): a profiler-sized case."""
    return adamw_2p30(26)


WORKLOADS = {
    "single": single_matrix,
    "gpt124m": gpt124m,
    "llama7b": llama7b,
    "llama7b_layer": llama7b_layer,
    "llama7b_bf16state": llama7b_bf16_state,
    "gpt124m_bf16state": gpt124m_bf16_state,
    "moe_mla": moe_mla,
    "moe_mla_e16": moe_mla_e16,
    "moe_mla_e16_cu": moe_mla_e16_cu,
    "adamw_2p26": adamw_2p26,
    "adamw_2p30": adamw_2p30,
}


# ---- materialisation -----------------------------------------------------------

def host_tensor(wl: Workload, kind: int, index: int, step: int = 0, offset: int = 0,
                count: int | None = None) -> np.ndarray:
    """Float64 copy (exact values of the stored dtype) of a tensor's inputs,
    or of ``count`` elements from flat ``offset``."""
    spec = (wl.muon if kind in (KIND_W, KIND_G) else wl.adamw)[index]
    n = spec.numel if count is None else count
    if kind in (KIND_W, KIND_AW):
        dt, std = spec.param_dtype, np.float32(spec.w_std)
        if getattr(spec, "w_const", None) is not None:
            return np.full(n, spec.w_const, dtype=np.float64)
    else:
        dt, std = spec.grad_dtype, wl.grad_std(kind, index)
    from . import normal
    return normal(wl.seed, tensor_id(kind, index, step if kind in (KIND_G, KIND_AG) else 0),
                  (n,), std=std, dtype=dt, offset=offset).astype(np.float64)


def device_tensor(wl: Workload, kind: int, index: int, step: int = 0, device="cuda"):
    """The same tensor created on the GPU by the CUDA generator."""
    import torch
    from .gpu import fill_normal
    spec = (wl.muon if kind in (KIND_W, KIND_G) else wl.adamw)[index]
    shape = spec.shape
    if kind in (KIND_W, KIND_AW):
        dt = spec.param_dtype
        tdt = torch.float32 if dt == "f32" else torch.bfloat16
        if getattr(spec, "w_const", None) is not None:
            return torch.full(shape, spec.w_const, dtype=tdt, device=device)
        t = torch.empty(shape, dtype=tdt, device=device)
        return fill_normal(t, wl.seed, tensor_id(kind, index), np.float32(spec.w_std))
    dt = spec.grad_dtype
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    t = torch.empty(shape, dtype=tdt, device=device)
    return fill_normal(t, wl.seed, tensor_id(kind, index, step), wl.grad_std(kind, index))
