"""Seeded synthetic inputs: random-init weights, token ids and pre-filled KV caches.

This module only draws random numbers; it holds none of the model's arithmetic. Both the CUDA
library's tests and the oracle's tests take their inputs from here, so the two sides see the same
bytes. Recipe (random init, no checkpoint): matrices bf16 N(0, 0.02); norm gains bf16
1 + U(-0.1, 0.1); token ids uniform in [0, vocab); pre-filled K/V bf16 N(0, 1). Each tensor has
its own seed, derived from the workload seed and the tensor's name, so any subset of layers can be
regenerated on its own.
"""
from __future__ import annotations

import zlib

import numpy as np
import torch

LAYER_NAMES = ("in_norm", "q_proj", "k_proj", "v_proj", "o_proj", "q_norm", "k_norm", "post_norm",
               "gate_proj", "up_proj", "down_proj")


def _seed(seed: int, name: str, layer: int = -1) -> int:
    return (seed * 1_000_003 + zlib.crc32(f"{name}:{layer}".encode())) & 0x7FFF_FFFF_FFFF


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std, seed, device):
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=_gen(device, seed))
    return t.to(torch.bfloat16)


def _gain(n, seed, device):
    t = torch.empty(n, dtype=torch.float32, device=device)
    t.uniform_(-0.1, 0.1, generator=_gen(device, seed))
    return (t + 1.0).to(torch.bfloat16)


def layer_shapes(cfg: dict) -> dict:
    d, dh, F = cfg["hidden"], cfg["head_dim"], cfg["intermediate"]
    qw, kvw = cfg["n_q_heads"] * dh, cfg["n_kv_heads"] * dh
    return {"in_norm": (d,), "q_proj": (qw, d), "k_proj": (kvw, d), "v_proj": (kvw, d),
            "o_proj": (d, qw), "q_norm": (dh,), "k_norm": (dh,), "post_norm": (d,),
            "gate_proj": (F, d), "up_proj": (F, d), "down_proj": (d, F)}


def make_layer(cfg: dict, seed: int, layer: int, device="cpu") -> dict:
    out = {}
    for name, shape in layer_shapes(cfg).items():
        s = _seed(seed, name, layer)
        out[name] = _gain(shape[0], s, device) if len(shape) == 1 else _normal(shape, 0.02, s, device)
    return out


def make_weights(cfg: dict, seed: int, device="cpu", layers=None) -> dict:
    """bf16 torch tensors. Per-layer entries are lists; layers not in ``layers`` are None."""
    d, V = cfg["hidden"], cfg["vocab"]
    w = {"embed": _normal((V, d), 0.02, _seed(seed, "embed"), device),
         "final_norm": _gain(d, _seed(seed, "final_norm"), device),
         "lm_head": None if cfg["tie_embeddings"] else _normal((V, d), 0.02, _seed(seed, "lm_head"), device)}
    keep = range(cfg["n_layers"]) if layers is None else layers
    for name in LAYER_NAMES:
        w[name] = [None] * cfg["n_layers"]
    for l in keep:
        for name, t in make_layer(cfg, seed, l, device).items():
            w[name][l] = t
    return w


def make_ids(vocab: int, batch: int, tokens: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(device, _seed(seed, "ids", batch * 1_000_000 + tokens))
    return torch.randint(0, vocab, (batch, tokens), generator=g, device=device, dtype=torch.int64).to(torch.int32)


def make_kv_normal(shape, seed: int, layer: int, which: str, device="cpu") -> torch.Tensor:
    return _normal(shape, 1.0, _seed(seed, "kv_" + which, layer), device)


def to_numpy_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> its uint16 bit patterns on the host (a view, no arithmetic)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_numpy_bits(a: np.ndarray, device="cpu") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def weights_to_numpy(w: dict) -> dict:
    out = {}
    for k, v in w.items():
        if isinstance(v, list):
            out[k] = [None if t is None else to_numpy_bits(t) for t in v]
        else:
            out[k] = None if v is None else to_numpy_bits(v)
    return out
