"""An fp64 statement of the Qwen3 forward pass written with PyTorch library routines
(matmul, rsqrt, silu, scaled_dot_product_attention with enable_gqa), following the pre-norm block of
"A modern architecture: Qwen3" (section The whole model) without any bf16 rounding. Used only to pin
the oracle's layer composition: the oracle must agree with it to within bf16 rounding noise.
"""
import torch
import torch.nn.functional as F


def forward_f64(cfg: dict, w: dict, ids: torch.Tensor) -> torch.Tensor:
    """w: bf16 torch tensors (synth.make_weights layout); ids [B, T]. Returns logits [B*T, V] fp64."""
    B, T = ids.shape
    hq, hkv, dh, eps = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"], cfg["rms_eps"]

    def rms(x, g):
        return g.double() * (x * torch.rsqrt(x.pow(2).mean(-1, keepdim=True) + eps))

    def rot(x):
        a, b = x.chunk(2, dim=-1)
        return torch.cat((-b, a), dim=-1)

    inv = cfg["rope_theta"] ** (-torch.arange(0, dh, 2, dtype=torch.float64) / dh)
    ang = torch.arange(T, dtype=torch.float64)[:, None] * inv
    ang = torch.cat((ang, ang), dim=-1)
    cos, sin = ang.cos(), ang.sin()
    x = w["embed"].double()[ids.long()]
    for l in range(cfg["n_layers"]):
        h = rms(x, w["in_norm"][l])
        q = (h @ w["q_proj"][l].double().T).view(B, T, hq, dh)
        k = (h @ w["k_proj"][l].double().T).view(B, T, hkv, dh)
        v = (h @ w["v_proj"][l].double().T).view(B, T, hkv, dh)
        q = rms(q, w["q_norm"][l]).transpose(1, 2)
        k = rms(k, w["k_norm"][l]).transpose(1, 2)
        v = v.transpose(1, 2)
        q, k = q * cos + rot(q) * sin, k * cos + rot(k) * sin
        o = F.scaled_dot_product_attention(q, k, v, is_causal=True, enable_gqa=True)
        x = x + o.transpose(1, 2).reshape(B, T, hq * dh) @ w["o_proj"][l].double().T
        h = rms(x, w["post_norm"][l])
        x = x + (F.silu(h @ w["gate_proj"][l].double().T) * (h @ w["up_proj"][l].double().T)) \
            @ w["down_proj"][l].double().T
    h = rms(x, w["final_norm"])
    head = w["embed"] if cfg["tie_embeddings"] else w["lm_head"]
    return (h @ head.double().T).reshape(B * T, -1)
