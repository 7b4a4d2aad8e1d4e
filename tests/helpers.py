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


def _update_base(wl: W.Workload, spec, W_prev):
    """The part of the new weight that is not the update: the decayed previous
    weight for the plain rule, the previous weight itself under a cautious
    mask (which gates the decay per element)."""
    hp = wl.muon_hp
    if hp.get("cautious", 0):
        return np.array(W_prev, dtype=np.float64)
    return (1.0 - hp["lr"] * spec.lr_mult * spec.wd) * np.asarray(W_prev, dtype=np.float64)


def _round_param(spec, W64):
    if spec.param_dtype == "f32":
        return W64.astype(np.float32).astype(np.float64)
    return oracle.round_bf16(W64)


def oracle_muon_tensor(wl: W.Workload, i: int, steps: int, views=None, keep_unrounded=False):
    """Oracle run of Muon tensor i for ``steps`` steps (fresh state).

    ``views`` restricts the run to a subset of the tensor's views (each view
    is independent). Returns a dict of the selected views stacked as
    (k, r, c): W (rounded to the param dtype), W64 (before that rounding), B,
    sm, U (the last step's update direction), base (the part of W64 that is
    not the last update) and B_atol (the running per-element bound on the
    fp32 momentum's rounding, tests.parity.momentum_atol)."""
    from tests.parity import momentum_atol
    spec = wl.muon[i]
    hp = oracle_hparams(wl)
    r, c = spec.rows, spec.cols
    sel = list(range(spec.views)) if views is None else list(views)
    out = {k: [] for k in ("W", "W64", "B", "sm", "U", "base", "B_atol")}
    for v in sel:
        off, cnt = v * r * c, r * c
        Wv = W.host_tensor(wl, W.KIND_W, i, offset=off, count=cnt).reshape(r, c)
        Bv = np.zeros((r, c))
        E = np.zeros((r, c))
        sm = np.zeros(r) if hp.normuon else None
        for s in range(steps):
            Gv = W.host_tensor(wl, W.KIND_G, i, step=s, offset=off, count=cnt).reshape(r, c)
            res = oracle.muon_step_view(Wv, Gv, Bv, hp, spec.lr_mult, spec.wd, sm)
            E = momentum_atol(Bv, Gv, hp.momentum, E)
            base = _update_base(wl, spec, Wv)
            W64 = res.W
            Wv = _round_param(spec, res.W)
            Bv, sm, U = res.B, res.sm, res.U
        for k, x in (("W", Wv), ("W64", W64), ("B", Bv), ("sm", sm), ("U", U), ("base", base),
                     ("B_atol", E)):
            out[k].append(x)
    res = {k: (None if out[k][0] is None else np.stack(out[k])) for k in out}
    res["views"] = sel
    return res


def oracle_muon_step_from(wl: W.Workload, i: int, step: int, views, W0, B0, sm0=None):
    """One oracle step of Muon tensor i from a given state: the device's own
    W, B (and NorMuon state) for the listed views, stacked (k, r, c), and the
    gradient of step index ``step``. Same keys as oracle_muon_tensor."""
    from tests.parity import momentum_atol
    spec = wl.muon[i]
    hp = oracle_hparams(wl)
    r, c = spec.rows, spec.cols
    out = {k: [] for k in ("W", "W64", "B", "sm", "U", "base", "B_atol")}
    for k, v in enumerate(views):
        off, cnt = v * r * c, r * c
        Gv = W.host_tensor(wl, W.KIND_G, i, step=step, offset=off, count=cnt).reshape(r, c)
        Wv = np.asarray(W0[k], dtype=np.float64)
        Bv = np.asarray(B0[k], dtype=np.float64)
        res = oracle.muon_step_view(Wv, Gv, Bv, hp, spec.lr_mult, spec.wd,
                                    None if sm0 is None else np.asarray(sm0[k], np.float64))
        for key, x in (("W", _round_param(spec, res.W)), ("W64", res.W), ("B", res.B),
                       ("sm", res.sm), ("U", res.U), ("base", _update_base(wl, spec, Wv)),
                       ("B_atol", momentum_atol(Bv, Gv, hp.momentum))):
            out[key].append(x)
    res = {k: (None if out[k][0] is None else np.stack(out[k])) for k in out}
    res["views"] = list(views)
    return res


def check_muon_views(wl: W.Workload, i: int, ref: dict, got_W, got_B, got_sm=None,
                     what: str = "", sm_bar: float = 4e-2) -> None:
    """Applies the parity bars of tests.parity to the views of ``ref``:
    momentum element by element, the parameter by its dtype's bars (one step
    from the state ``ref`` started from), the NorMuon state at ``sm_bar``."""
    from tests.parity import check_bf16_param, check_f32_update, check_fp32
    spec = wl.muon[i]
    hp = oracle_hparams(wl)
    step_scale = hp.lr * spec.lr_mult * oracle.shape_scale(spec.rows, spec.cols, hp.shape_rule)
    for k, v in enumerate(ref["views"]):
        tag = f"{what or wl.name}:{spec.name}[{v}]"
        check_fp32(got_B[k], ref["B"][k], ref["B_atol"][k], tag + " momentum")
        if spec.param_dtype == "bf16":
            check_bf16_param(got_W[k], ref["W64"][k], ref["base"][k], step_scale, ref["U"][k],
                             tag + " param")
        else:
            check_f32_update(got_W[k], ref["W64"][k], ref["base"][k], tag + " param")
        if got_sm is not None and ref["sm"] is not None:
            err = rel_fro(got_sm[k], ref["sm"][k])
            assert err < sm_bar, (tag, "NorMuon state", err)


def oracle_adam_tensor(wl: W.Workload, j: int, steps: int, offset: int = 0, count=None):
    """Oracle run of AdamW tensor j (a slice of it) for ``steps`` steps, with
    the running per-element bounds (m_atol, v_atol, W_atol) of
    tests.parity.adamw_atol."""
    from tests.parity import adamw_atol
    spec = wl.adamw[j]
    n = spec.numel if count is None else count
    hp = wl.adam_hp
    Wt = W.host_tensor(wl, W.KIND_AW, j, offset=offset, count=n)
    m = np.zeros(n)
    v = np.zeros(n)
    E = (0.0, 0.0, 0.0)
    lr = hp["lr"] * spec.lr_mult
    for s in range(steps):
        G = W.host_tensor(wl, W.KIND_AG, j, step=s, offset=offset, count=n)
        E = adamw_atol(Wt, G, m, v, lr, hp["betas"][0], hp["betas"][1], hp["eps"], spec.wd, s + 1,
                       E)
        Wt, m, v = oracle.adamw_step(Wt, G, m, v, lr, hp["betas"][0],
                                     hp["betas"][1], hp["eps"], spec.wd, s + 1)
        Wt = oracle.round_bf16(Wt) if spec.param_dtype == "bf16" else \
            Wt.astype(np.float32).astype(np.float64)
    return dict(W=Wt, m=m, v=v, m_atol=E[0], v_atol=E[1], W_atol=E[2])


def oracle_adam_step_from(wl: W.Workload, j: int, step: int, offset: int, count: int, W0, m0, v0):
    """One oracle AdamW step of a slice of tensor j from a given state (the
    device's own W, m, v) with the gradient of step index ``step`` (bias
    correction t = step + 1); same keys as oracle_adam_tensor."""
    from tests.parity import adamw_atol
    spec = wl.adamw[j]
    hp = wl.adam_hp
    lr = hp["lr"] * spec.lr_mult
    G = W.host_tensor(wl, W.KIND_AG, j, step=step, offset=offset, count=count)
    Wt, m, v = (np.asarray(x, dtype=np.float64) for x in (W0, m0, v0))
    E = adamw_atol(Wt, G, m, v, lr, hp["betas"][0], hp["betas"][1], hp["eps"], spec.wd, step + 1)
    Wn, m, v = oracle.adamw_step(Wt, G, m, v, lr, hp["betas"][0], hp["betas"][1], hp["eps"],
                                 spec.wd, step + 1)
    Wn = oracle.round_bf16(Wn) if spec.param_dtype == "bf16" else \
        Wn.astype(np.float32).astype(np.float64)
    return dict(W=Wn, m=m, v=v, m_atol=E[0], v_atol=E[1], W_atol=E[2])


def check_adam_result(got_W, got_m, got_v, ref: dict, param_dtype: str, what: str,
                      steps: int = 1) -> None:
    """AdamW parity: moments element by element (tests.parity.check_fp32); an
    fp32 parameter the same way; a bf16 parameter at most one bf16 spacing
    from the oracle's rounded value. The fp32 error before the rounding is far
    below a spacing, so only values within that error of a rounding boundary
    can land one spacing away: the count of such elements may not exceed
    max(3, 2x) their expected number, sum(min(1, 2 SAFETY W_atol / ulp)).
    After ``steps`` > 1 steps run independently on both sides, a bf16
    parameter is held to 1e-3 relative Frobenius instead: each step's flips
    persist (the update does not depend on the weight), and an element that
    shrinks across binades carries a flip made at a larger magnitude as
    several spacings of its final value; the one-step bars above apply to a
    step taken from the device's own state."""
    from tests.parity import bf16_ulp, check_fp32, record
    check_fp32(got_m, ref["m"], ref["m_atol"], what + " m")
    check_fp32(got_v, ref["v"], ref["v_atol"], what + " v")
    if param_dtype == "f32":
        check_fp32(got_W, ref["W"], ref["W_atol"], what + " W")
        return
    from tests.parity import SAFETY
    got = np.asarray(got_W, dtype=np.float64)
    want = ref["W"]
    if steps > 1:
        err = rel_fro(got, want)
        record("bf16_adamw_drift", what, n=int(want.size), steps=steps, w_rel=err)
        assert err < 1e-3, (what, err)
        return
    ulp = bf16_ulp(want)
    diff = np.abs(got - want)
    flips = int(np.sum(diff > 0))
    expected = float(np.sum(np.minimum(1.0, 2 * SAFETY * np.broadcast_to(ref["W_atol"],
                                                                           want.shape) / ulp)))
    record("bf16_adamw_param", what, n=int(want.size), flips=flips, flips_expected=expected,
           max_ulps=float(np.max(diff / ulp)) if want.size else 0.0)
    assert np.all(diff <= ulp), (what, float(np.max(diff / ulp)))
    assert flips <= max(3.0, 2.0 * expected), (what, flips, expected)


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
