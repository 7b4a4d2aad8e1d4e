"""Host-side Muon / AdamW parameter split (not part of the timed step).

Speedtronic docs "v2 optimizers", "Hybrid routing": Muon takes hidden 2-D
matrix weights (attention Q/K/V/output, MLP gate/up/down, neutral 2-D
matrices); AdamW keeps embeddings and positional embeddings, LM heads,
classifiers and output projections, normalisation parameters, biases,
scalars, non-2-D tensors and frozen parameters. A parameter appears once
(tied weights are deduplicated; kimi-k3 "Optimization": every trainable
parameter is assigned once). Matrix views (kimi-k3, "A tensor's storage
shape can be misleading") are declared by the caller per parameter name.
"""
from __future__ import annotations

ADAMW_NAME_HINTS = ("embed", "wte", "wpe", "pos_emb", "lm_head", "head", "classifier",
                    "output_proj", "norm", "ln_", "bias", "scale")


def _is_adamw_name(name: str) -> bool:
    leaf = name.lower()
    return any(h in leaf for h in ADAMW_NAME_HINTS)


def route_parameters(named_parameters, views: dict | None = None, roles: dict | None = None):
    """Split ``(name, tensor)`` pairs into Muon and AdamW lists.

    ``views`` maps a parameter name to its number of matrix views (default 1).
    ``roles`` maps a name to "muon" or "adamw" and overrides the heuristic; a
    "muon" role is only valid for a floating-point 2-D (or viewed) parameter.
    Returns (muon, adamw): lists of (name, tensor, views) and (name, tensor).
    """
    views = views or {}
    roles = roles or {}
    seen = set()
    muon, adamw = [], []
    for name, p in named_parameters:
        key = id(p)
        if key in seen:
            continue
        seen.add(key)
        role = roles.get(name)
        if role is not None and role not in ("muon", "adamw"):
            raise ValueError(f"{name}: role must be 'muon' or 'adamw', not {role!r}")
        floating = getattr(p, "is_floating_point", lambda: True)()
        is_matrix = p.dim() == 2 or (p.dim() == 3 and name in views)
        if role == "muon":
            if not (floating and is_matrix and getattr(p, "requires_grad", True)):
                raise ValueError(f"{name}: the muon role needs a trainable floating 2-D parameter")
            muon.append((name, p, int(views.get(name, p.shape[0] if p.dim() == 3 else 1))))
        elif (role == "adamw" or not floating or not is_matrix or _is_adamw_name(name)
              or not getattr(p, "requires_grad", True)):
            adamw.append((name, p))
        else:
            muon.append((name, p, int(views.get(name, p.shape[0] if p.dim() == 3 else 1))))
    return muon, adamw
