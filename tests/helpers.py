"""Shared test helpers: run a synthetic workload through the C ABI on the GPU,
and through the fp64 oracle on the CPU, on identical seeded inputs."""
from __future__ import annotations

import numpy as np

import oracle
from synth import workloads as W


def rel_fro(got, want) -> float:
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.linalg.norm(want)
    num = np.linalg.norm(got - want)
    return float(num / den) if den > 0 else float(num)


def to_np(t) -> np.ndarray:
    import torch
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_hparams(wl: W.Workload) -> oracle.MuonHparams:
    hp = wl.muon_hp
    return oracle.MuonHparams(lr=hp["lr"], momentum=hp["momentum"], nesterov=hp["nesterov"],
                              eps=hp["eps"], ns_steps=hp["ns_steps"], coeffs=tuple(hp["coeffs"]),
                              norm_scale=hp.get("norm_scale", 1.0),
                              normuon=hp.get("normuon", False), beta2=hp.get("beta2", 0.95),
                              muon_plus=hp.get("muon_plus", False),
                              plus_eps=hp.get("plus_eps", hp["eps"]),
                              cautious=hp.get("cautious", 0),
                              normuon_eps=hp.get("normuon_eps", oracle.NORMUON_FLOOR),
                              shape_rule=hp.get("shape_rule", oracle.SHAPE_RATIO))


def oracle_muon_tensor(wl: W.Workload, i: int, steps: int, views=None, keep_unrounded=False):
    """Oracle run of Muon tensor i for ``steps`` steps (fresh state).

    ``views`` restricts the run to a subset of the tensor's views (each view
    is independent). Returns dict of W (rounded to the param dtype), B, sm, U
    for the selected views stacked as (k, r, c)."""
    spec = wl.muon[i]
    hp = oracle_hparams(wl)
    r, c = spec.rows, spec.cols
    sel = list(range(spec.views)) if views is None else list(views)
    out_W, out_B, out_sm, out_U, out_W64 = [], [], [], [], []
    for v in sel:
        off, cnt = v * r * c, r * c
        Wv = W.host_tensor(wl, W.KIND_W, i, offset=off, count=cnt).reshape(r, c)
        Bv = np.zeros((r, c))
        sm = np.zeros(r) if hp.normuon else None
        U = None
        for s in range(steps):
            Gv = W.host_tensor(wl, W.KIND_G, i, step=s, offset=off, count=cnt).reshape(r, c)
            res = oracle.muon_step_view(Wv, Gv, Bv, hp, spec.lr_mult, spec.wd, sm)
            W64 = res.W
            Wv = res.W if spec.param_dtype == "f32" else oracle.round_bf16(res.W)
            if spec.param_dtype == "f32":
                Wv = Wv.astype(np.float32).astype(np.float64)
            Bv, sm, U = res.B, res.sm, res.U
        out_W.append(Wv)
        out_W64.append(W64)
        out_B.append(Bv)
        out_sm.append(sm)
        out_U.append(U)
    return dict(W=np.stack(out_W), W64=np.stack(out_W64), B=np.stack(out_B), U=np.stack(out_U),
                sm=None if out_sm[0] is None else np.stack(out_sm), views=sel)


def oracle_adam_tensor(wl: W.Workload, j: int, steps: int, offset: int = 0, count=None):
    spec = wl.adamw[j]
    n = spec.numel if count is None else count
    hp = wl.adam_hp
    Wt = W.host_tensor(wl, W.KIND_AW, j, offset=offset, count=n)
    m = np.zeros(n)
    v = np.zeros(n)
    for s in range(steps):
        G = W.host_tensor(wl, W.KIND_AG, j, step=s, offset=offset, count=n)
        Wt, m, v = oracle.adamw_step(Wt, G, m, v, hp["lr"] * spec.lr_mult, hp["betas"][0],
                                     hp["betas"][1], hp["eps"], spec.wd, s + 1)
        Wt = oracle.round_bf16(Wt) if spec.param_dtype == "bf16" else \
            Wt.astype(np.float32).astype(np.float64)
    return dict(W=Wt, m=m, v=v)


class DeviceRun:
    """A workload's tensors on the GPU, stepped through the C ABI."""

    def __init__(self, wl: W.Workload, device="cuda"):
        import torch
        import muon_adamw_hybrid_gb300 as mh
        self.wl, self.mh, self.torch = wl, mh, torch
        hp = wl.muon_hp
        self.hp = mh.make_hparams(lr=hp["lr"], momentum=hp["momentum"], nesterov=hp["nesterov"],
                                  eps=hp["eps"], ns_steps=hp["ns_steps"], coeffs=hp["coeffs"],
                                  norm_scale=hp.get("norm_scale", 1.0),
                                  normuon=hp.get("normuon", False), beta2=hp.get("beta2", 0.95),
                                  muon_plus=hp.get("muon_plus", False),
                                  plus_eps=hp.get("plus_eps", hp["eps"]),
                                  cautious=hp.get("cautious", 0),
                                  normuon_eps=hp.get("normuon_eps", oracle.NORMUON_FLOOR),
                                  shape_rule=hp.get("shape_rule", 0))
        self.mW = [W.device_tensor(wl, W.KIND_W, i, device=device) for i in range(len(wl.muon))]
        self.mG = [W.device_tensor(wl, W.KIND_G, i, 0, device=device) for i in range(len(wl.muon))]
        self.mB = [torch.zeros(s.shape, dtype=torch.float32, device=device) for s in wl.muon]
        self.sm = [torch.zeros(s.views * s.rows, dtype=torch.float32, device=device)
                   if self.hp.normuon else None for s in wl.muon]
        self.aW = [W.device_tensor(wl, W.KIND_AW, j, device=device) for j in range(len(wl.adamw))]
        self.aG = [W.device_tensor(wl, W.KIND_AG, j, 0, device=device) for j in range(len(wl.adamw))]
        self.am = [torch.zeros(s.shape, dtype=torch.float32, device=device) for s in wl.adamw]
        self.av = [torch.zeros(s.shape, dtype=torch.float32, device=device) for s in wl.adamw]
        self.ts = [mh.muon_tensor(w, g, b, s.views, sm, s.lr_mult, s.wd)
                   for w, g, b, sm, s in zip(self.mW, self.mG, self.mB, self.sm, wl.muon)]
        self.at = [mh.adamw_tensor(w, g, m, v, s.lr_mult, s.wd)
                   for w, g, m, v, s in zip(self.aW, self.aG, self.am, self.av, wl.adamw)]
        need = mh.muon_workspace_bytes(self.ts, self.hp) if self.ts else 0
        self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        self.step_count = 0

    def refresh_grads(self, step: int) -> None:
        from synth.gpu import fill_normal
        wl = self.wl
        for i, g in enumerate(self.mG):
            fill_normal(g, wl.seed, W.tensor_id(W.KIND_G, i, step), wl.grad_std(W.KIND_G, i))
        for j, g in enumerate(self.aG):
            fill_normal(g, wl.seed, W.tensor_id(W.KIND_AG, j, step), wl.grad_std(W.KIND_AG, j))

    def step(self) -> None:
        mh, torch = self.mh, self.torch
        s = torch.cuda.current_stream().cuda_stream
        if self.step_count > 0:
            self.refresh_grads(self.step_count)
        self.step_count += 1
        if self.ts:
            mh.muon_step_batched(self.ts, self.hp, self.ws.data_ptr(), self.ws.numel(), s)
        if self.at:
            hp = self.wl.adam_hp
            mh.adamw_step(self.at, hp["lr"], hp["betas"][0], hp["betas"][1], hp["eps"],
                          self.step_count, s)

    def status_ok(self) -> None:
        s = self.torch.cuda.current_stream().cuda_stream
        self.mh.workspace_status(self.ws.data_ptr(), s)
