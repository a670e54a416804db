"""Pins for the oracle's operations: the pages' worked examples, closed forms, invariants, and
independent library routines (PyTorch CPU bf16/fp64 arithmetic, scaled_dot_product_attention).

Every check lives in a ``check_*`` function so that tests/test_oracle_planted.py can rerun the
same checks against oracle builds with a planted mistake and show that one of them fails.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O
from qwen3_decoder_transformer_gb300 import QWEN3_0P6B, QWEN3_8B, synth
from tests.conftest import read_golden

bits, frm = synth.to_numpy_bits, synth.from_numpy_bits


def _rot_half(x):
    a, b = x.chunk(2, dim=-1)
    return torch.cat((-b, a), dim=-1)


# ------------------------------------------------------------------------------- bf16 conversion

def check_bf16_conversion():
    one = 1.0
    assert O.bf16_from_f32(np.float32(one)) == 0x3F80
    # exact ties go to even: 1 + 2^-8 -> 1.0 ; 1 + 3*2^-8 -> 1 + 2^-6
    assert O.bf16_from_f32(np.float32(1 + 2 ** -8)) == 0x3F80
    assert O.bf16_from_f32(np.float32(1 + 3 * 2 ** -8)) == 0x3F82
    assert O.bf16_from_f32(np.float32(np.inf)) == 0x7F80
    assert O.bf16_from_f32(np.float32(np.nan)) & 0x7FC0 == 0x7FC0
    # double -> bf16 is one rounding: just above a tie rounds up even where float(x) is the tie
    assert O.bf16_from_f64(1 + 2 ** -8 + 2 ** -40) == 0x3F81
    assert O.bf16_from_f64(1 + 2 ** -8) == 0x3F80
    assert O.bf16_from_f64(-(1 + 2 ** -8 + 2 ** -40)) == 0xBF81
    # agreement with PyTorch's float -> bfloat16 on random values
    x = torch.randn(4096) * torch.logspace(-20, 20, 4096)
    assert np.array_equal(O.bf16_from_f32(x.numpy()), bits(x.to(torch.bfloat16)))


def test_bf16_conversion():
    check_bf16_conversion()


# ------------------------------------------------------------------------------------- RMSNorm

def check_rmsnorm_worked_example():
    g = read_golden("rmsnorm_worked_example.txt")
    y = O.rmsnorm_core_f32(np.array(g["input"], dtype=np.float32), 0.0)
    assert np.round(y.astype(np.float64), int(g["decimals"])).tolist() == g["output"]
    x = np.array(g["input"], dtype=np.float64)
    assert round(math.sqrt((x ** 2).mean()), 4) == g["rms"]


def check_rmsnorm_invariants():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(1000).astype(np.float32) * 7
    y = O.rmsnorm_core_f32(x, 0.0).astype(np.float64)
    assert abs((y ** 2).mean() - 1.0) < 1e-5  # unit RMS
    y2 = O.rmsnorm_core_f32((x * 16).astype(np.float32), 0.0).astype(np.float64)
    assert np.allclose(y, y2, rtol=1e-6, atol=0)  # scale invariant (power-of-two scale is exact)
    assert np.all(np.sign(y) == np.sign(x))  # direction unchanged


def check_rmsnorm_bf16_pages_order():
    """The pages' fp32-reduce, cast-to-input-dtype, then times-gamma order, run by PyTorch."""
    torch.manual_seed(0)
    eps = 1e-6
    x = (torch.randn(64, 256) * 3).to(torch.bfloat16)
    gam = (1 + 0.2 * (torch.rand(256) - 0.5)).to(torch.bfloat16)
    x32 = x.float()
    ref = gam * (x32 * torch.rsqrt(x32.square().mean(-1, keepdim=True) + eps)).to(torch.bfloat16)
    got = O.rmsnorm(bits(x), bits(gam), eps)
    assert np.array_equal(got, bits(ref))


def test_rmsnorm_worked_example():
    check_rmsnorm_worked_example()


def test_rmsnorm_invariants():
    check_rmsnorm_invariants()


def test_rmsnorm_bf16_pages_order():
    check_rmsnorm_bf16_pages_order()


# ------------------------------------------------------------------------------------- linear

def check_linear():
    rng = np.random.default_rng(2)
    a = torch.from_numpy(rng.standard_normal((7, 96))).to(torch.bfloat16)
    w = torch.from_numpy(rng.standard_normal((40, 96)) * 0.05).to(torch.bfloat16)
    ref = (a.double() @ w.double().T)
    got = O.f32_from_bf16(O.linear(bits(a), bits(w))).astype(np.float64)
    # one rounding to bf16: within half an ulp (2^-8 relative) of the exact product
    assert np.all(np.abs(got - ref.numpy()) <= 2.0 ** -8 * np.abs(ref.numpy()) + 1e-30)
    got32 = O.linear(bits(a), bits(w), f32_out=True).astype(np.float64)
    assert np.allclose(got32, ref.numpy(), rtol=2e-7, atol=1e-30)


def test_linear():
    check_linear()


def check_residual_add():
    torch.manual_seed(11)
    x = (torch.randn(5000) * 4).to(torch.bfloat16)
    y = (torch.randn(5000) * torch.logspace(-6, 2, 5000)).to(torch.bfloat16)
    assert np.array_equal(O.residual_add(bits(x), bits(y)), bits(x + y))


def test_residual_add():
    check_residual_add()


# --------------------------------------------------------------------------------- SiLU/SwiGLU

def check_silu_worked_example():
    g = read_golden("silu_worked_example.txt")
    d = int(g["decimals"])
    assert round(O.silu(0.0), d) == g["silu_0"]
    assert round(O.silu(2.0), d) == g["silu_2"]
    assert round(O.silu(2.0) * g["up"], d) == g["passed"]


def check_swiglu_bf16():
    torch.manual_seed(3)
    gg = (torch.randn(20000) * 3).to(torch.bfloat16)
    uu = torch.randn(20000).to(torch.bfloat16)
    assert np.array_equal(O.swiglu(bits(gg), bits(uu)), bits(F.silu(gg) * uu))


def test_silu_worked_example():
    check_silu_worked_example()


def test_swiglu_bf16():
    check_swiglu_bf16()


# --------------------------------------------------------------------------------------- RoPE

def check_rope_worked_example():
    g = read_golden("rope_relative_score.txt")
    q, k = np.array(g["q"]), np.array(g["k"])
    om = np.array([g["omega"]])
    p = g["pairs"]
    for i in range(0, len(p), 2):
        s = O.rope_rotate_f64(q, p[i], om) @ O.rope_rotate_f64(k, p[i + 1], om)
        assert round(s, int(g["decimals"])) == g["score"]


def check_rope_identities():
    rng = np.random.default_rng(4)
    dim = 128
    om = O.rope_inv_freq(1e6, dim).astype(np.float64)
    q, k = rng.standard_normal(dim), rng.standard_normal(dim)
    # norm preserved
    assert abs(np.linalg.norm(O.rope_rotate_f64(q, 977, om)) - np.linalg.norm(q)) < 1e-10
    # distance 0 scores the plain dot product
    assert abs(O.rope_rotate_f64(q, 321, om) @ O.rope_rotate_f64(k, 321, om) - q @ k) < 1e-10
    # (R(p w) q) . (R(s w) k) = q^T R((s-p) w) k: depends on s - p only
    a = O.rope_rotate_f64(q, 5, om) @ O.rope_rotate_f64(k, 12, om)
    b = O.rope_rotate_f64(q, 105, om) @ O.rope_rotate_f64(k, 112, om)
    c = q @ O.rope_rotate_f64(k, 7, om)
    assert abs(a - b) < 1e-9 and abs(a - c) < 1e-9
    # 2x2 case: R(a)^T R(b) = R(b - a), applied to the basis vectors
    for e in (np.array([1.0, 0.0]), np.array([0.0, 1.0])):
        lhs = O.rope_rotate_f64(O.rope_rotate_f64(e, 0.9, np.array([1.0])), -0.4, np.array([1.0]))
        assert np.allclose(lhs, O.rope_rotate_f64(e, 0.5, np.array([1.0])), atol=1e-14)
    # R(phi) = [[cos, -sin], [sin, cos]]: e0 -> (cos, sin)
    assert np.allclose(O.rope_rotate_f64(np.array([1.0, 0.0]), 0.3, np.array([1.0])),
                       [math.cos(0.3), math.sin(0.3)], atol=1e-15)


def check_rope_frequencies():
    g = read_golden("rope_frequency_extremes.txt")
    inv = O.rope_inv_freq(g["theta"], int(g["dim"]))
    assert inv[0] == g["fastest"]
    assert abs(inv[-1] / g["slowest_about"] - 1) < 0.05
    assert abs(2 * math.pi / inv[-1] / g["wavelength_about"] - 1) < 0.05
    assert np.all(np.diff(inv) < 0)
    # each entry is theta^(-2i/d) correctly rounded to fp32
    i = np.arange(inv.size)
    exact = g["theta"] ** (-2.0 * i / g["dim"])
    assert np.array_equal(inv, exact.astype(np.float32))


def check_rope_bf16_pages_formula():
    """x * cos + rotate_half(x) * sin with bf16 tables, as the pages' PyTorch code evaluates it."""
    dim = 128
    inv = O.rope_inv_freq(1e6, dim)
    pos = torch.tensor([0, 1, 2, 7, 100, 4095, 4096, 32767, 32831])
    ang = pos.float()[:, None] * torch.from_numpy(inv)
    ang = torch.cat((ang, ang), dim=-1)
    cos, sin = ang.cos().to(torch.bfloat16), ang.sin().to(torch.bfloat16)
    torch.manual_seed(5)
    x = torch.randn(len(pos), dim).to(torch.bfloat16)
    ref = x * cos + _rot_half(x) * sin
    for i, p in enumerate(pos.tolist()):
        c, s = O.rope_cos_sin(p, inv)
        assert np.array_equal(c, bits(cos[i, :dim // 2])) and np.array_equal(s, bits(sin[i, :dim // 2]))
        assert np.array_equal(O.rope_apply(bits(x[i]), c, s), bits(ref[i]))


def test_rope_worked_example():
    check_rope_worked_example()


def test_rope_identities():
    check_rope_identities()


def test_rope_frequencies():
    check_rope_frequencies()


def test_rope_bf16_pages_formula():
    check_rope_bf16_pages_formula()


# ---------------------------------------------------------------------------------- attention

def check_gqa_attention_vs_sdpa():
    g = read_golden("gqa_attention_check.txt")
    hq, hkv, T, dh = int(g["q_heads"]), int(g["kv_heads"]), int(g["tokens"]), int(g["head_size"])
    torch.manual_seed(6)
    q = torch.randn(1, hq, T, dh).to(torch.bfloat16)
    k = torch.randn(1, hkv, T, dh).to(torch.bfloat16)
    v = torch.randn(1, hkv, T, dh).to(torch.bfloat16)
    ref = F.scaled_dot_product_attention(q.double(), k.double(), v.double(), is_causal=True,
                                         enable_gqa=True)[0]
    kc, vc = bits(k[0]), bits(v[0])  # cache set [Hkv][cap=T][dh]
    got = np.stack([O.attention_gqa_row_f64(bits(q[0, :, t]), kc, vc, t + 1) for t in range(T)], 1)
    assert np.max(np.abs(got - ref.numpy())) < 1e-12
    # row 0 sees only key 0: output = v0 of its kv head
    v0 = O.f32_from_bf16(vc[:, 0]).astype(np.float64)
    assert np.array_equal(got[:, 0], v0[np.arange(hq) // (hq // hkv)])


def test_gqa_attention_vs_sdpa():
    check_gqa_attention_vs_sdpa()


# ------------------------------------------------------------------------------- param counts

def check_param_count_0p6b():
    g = read_golden("qwen3_0p6b_param_count.txt")
    got = O.param_count(QWEN3_0P6B)
    for key in ("embedding", "attention", "qk_norm", "feed_forward", "other_norms"):
        assert got[key] == g[key], key
    assert sum(got.values()) == g["total"]


def check_param_count_8b():
    g = read_golden("qwen3_8b_model_card.txt")
    got = O.param_count(QWEN3_8B)
    total = sum(got.values())
    assert round(total / 1e9, 1) == g["params_billion"]
    assert round((total - got["embedding"] - got["lm_head"]) / 1e9, 2) == g["non_embedding_billion"]
    assert QWEN3_8B["n_layers"] == g["layers"] and QWEN3_8B["n_q_heads"] == g["q_heads"]
    assert QWEN3_8B["n_kv_heads"] == g["kv_heads"]


def test_param_count_0p6b():
    check_param_count_0p6b()


def test_param_count_8b():
    check_param_count_8b()


ALL_CHECKS = [check_bf16_conversion, check_rmsnorm_worked_example, check_rmsnorm_invariants,
              check_rmsnorm_bf16_pages_order, check_linear, check_residual_add, check_silu_worked_example,
              check_swiglu_bf16, check_rope_worked_example, check_rope_identities,
              check_rope_frequencies, check_rope_bf16_pages_formula, check_gqa_attention_vs_sdpa,
              check_param_count_0p6b, check_param_count_8b]
