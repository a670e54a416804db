"""The bench's roofline numerators against facts from outside the bench.

* GEMM FLOPs: two FLOPs per weight and token, so one token's projections must cost twice the
  parameter table of "Transformer architectures: modern" (section 6, Qwen3-0.6B: attention and
  feed-forward weights, tied embedding for the LM head) exactly, and twice the 8B model card's
  6.95B non-embedding parameters to within the norms' share.
* Attention FLOPs: 4 * head_dim per visible (query, key) pair and query head, the pairs counted by
  brute force over a causal mask.
* The `traffic` field: a profile summary counts only while the hash it records matches the kernel
  source; a changed or missing summary gives None.
"""
import hashlib
import importlib.util
import os

import numpy as np
import pytest

from qwen3_decoder_transformer_gb300.configs import QWEN3_0P6B, QWEN3_8B
from tests.conftest import ROOT, read_golden


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


GEMMS = ("gemm_qkv_norm_rope_append", "gemm_o_residual", "gemm_gateup_swiglu", "gemm_down_residual")


def test_gemm_flops_match_the_0p6b_parameter_table(bench):
    g = read_golden("qwen3_0p6b_param_count.txt")
    w = bench.kernel_work(QWEN3_0P6B, 1, 1)  # one token
    per_token = QWEN3_0P6B["n_layers"] * sum(w[k][1] for k in GEMMS)
    assert per_token == 2 * (g["attention"] + g["feed_forward"])
    assert w["gemm_lmhead"][1] == 2 * g["embedding"]  # tied head: the embedding matrix


def test_gemm_flops_match_the_8b_model_card(bench):
    g = read_golden("qwen3_8b_model_card.txt")
    w = bench.kernel_work(QWEN3_8B, 1, 1)
    per_token = QWEN3_8B["n_layers"] * sum(w[k][1] for k in GEMMS)
    # the card's non-embedding count also holds the norm gains (about 0.3M of 6.95B)
    assert abs(per_token / (2 * g["non_embedding_billion"] * 1e9) - 1) < 2e-3


@pytest.mark.parametrize("B,T,hq,dh", [(1, 1, 1, 8), (2, 37, 3, 8), (1, 130, 2, 64)])
def test_attention_flops_count_causal_pairs(bench, B, T, hq, dh):
    cfg = dict(hidden=hq * dh, head_dim=dh, intermediate=8, vocab=8, n_q_heads=hq, n_kv_heads=1, n_layers=1)
    visible = int(np.tril(np.ones((T, T), dtype=np.int64)).sum())  # key <= query
    assert bench.kernel_work(cfg, B, T)["attn_prefill"][1] == 4 * dh * visible * hq * B


def test_step_flops_sum_the_layers_and_the_head(bench):
    w = bench.kernel_work(QWEN3_8B, 1, 4096)
    per_layer = sum(w[k][1] for k in GEMMS) + w["attn_prefill"][1]
    assert bench.step_flops(QWEN3_8B, 1, 4096) == QWEN3_8B["n_layers"] * per_layer + w["gemm_lmhead"][1]


def test_traffic_counts_only_a_current_profile(bench, tmp_path, monkeypatch):
    src = tmp_path / "qwen3_decoder_transformer_gb300" / "csrc" / "attention.cu"
    src.parent.mkdir(parents=True)
    src.write_text("// kernel source\n")
    prof = tmp_path / "profiles" / "attn_prefill_some-workload.md"
    prof.parent.mkdir()
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    prof.write_text(f"source_sha256: {sha} (when captured)\n- traffic_bytes_per_launch: 123456\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profiles("attn_prefill", "some-workload") == 123456.0
    assert bench.traffic_from_profiles("attn_prefill", "other-workload") is None
    src.write_text("// kernel source, changed\n")
    assert bench.traffic_from_profiles("attn_prefill", "some-workload") is None
