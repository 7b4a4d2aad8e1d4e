"""Host-side Muon / AdamW routing (Speedtronic "v2 optimizers", "Hybrid routing")."""
import pytest
import torch

from muon_adamw_hybrid_gb300 import route_parameters


def _p(*shape, grad=True, dtype=torch.float32):
    return torch.zeros(*shape, dtype=dtype).requires_grad_(grad)


def test_default_split():
    emb = _p(100, 16)
    named = [("embed_tokens.weight", emb), ("layers.0.attn.q_proj.weight", _p(16, 16)),
             ("layers.0.attn.o_proj.weight", _p(16, 16)), ("layers.0.mlp.down.weight", _p(16, 64)),
             ("layers.0.input_norm.weight", _p(16)), ("layers.0.mlp.up.bias", _p(64)),
             ("lm_head.weight", _p(100, 16)), ("scalar_gate", _p(())),
             ("frozen.weight", _p(16, 16, grad=False)), ("tied_head.weight", emb),
             ("experts.gate_up", _p(4, 32, 16))]
    muon, adamw = route_parameters(named, views={"experts.gate_up": 4})
    assert [(n, v) for n, _, v in muon] == [("layers.0.attn.q_proj.weight", 1),
                                            ("layers.0.attn.o_proj.weight", 1),
                                            ("layers.0.mlp.down.weight", 1),
                                            ("experts.gate_up", 4)]
    names = [n for n, _ in adamw]
    assert names == ["embed_tokens.weight", "layers.0.input_norm.weight", "layers.0.mlp.up.bias",
                     "lm_head.weight", "scalar_gate", "frozen.weight"]
    # the tied head is the embedding object: assigned once
    assert "tied_head.weight" not in names


def test_role_override():
    muon, adamw = route_parameters([("lm_head.weight", _p(8, 8)), ("w", _p(8, 8))],
                                   roles={"lm_head.weight": "muon", "w": "adamw"})
    assert [n for n, _, _ in muon] == ["lm_head.weight"]
    assert [n for n, _ in adamw] == ["w"]


def test_invalid_roles_raise():
    with pytest.raises(ValueError):
        route_parameters([("b", _p(8))], roles={"b": "muon"})
    with pytest.raises(ValueError):
        route_parameters([("w", _p(8, 8))], roles={"w": "sgd"})
    with pytest.raises(ValueError):
        route_parameters([("w", _p(8, 8, dtype=torch.int32, grad=False))], roles={"w": "muon"})
