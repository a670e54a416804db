"""The seeded synthetic inputs follow the recipe the workloads are built from: weight matrices bf16
N(0, 0.02), norm gains bf16 1 + U(-0.1, 0.1), token ids uniform in [0, vocab), pre-filled K/V bf16
N(0, 1); each tensor seeded from the workload seed and its own name, so the same seed gives the same
bytes (the CUDA path and the oracle see identical inputs) and layers can be regenerated alone."""
import numpy as np
import pytest
import torch

from qwen3_decoder_transformer_gb300 import synth
from qwen3_decoder_transformer_gb300.configs import QWEN3_0P6B, QWEN3_8B


def _f(t):
    return t.float().numpy().astype(np.float64)


@pytest.mark.parametrize("cfg", [QWEN3_0P6B, QWEN3_8B])
def test_layer_shapes_and_distributions(cfg):
    layer = synth.make_layer(cfg, seed=5, layer=3)
    assert {k: tuple(v.shape) for k, v in layer.items()} == synth.layer_shapes(cfg)
    for name, t in layer.items():
        assert t.dtype == torch.bfloat16, name
        x = _f(t)
        if t.dim() == 1:  # norm gain: 1 + U(-0.1, 0.1), rounded to bf16 (half a step: 2^-9 below 1, 2^-8 above)
            assert x.min() >= 0.9 - 2.0**-9 and x.max() <= 1.1 + 2.0**-8, name
            assert abs(x.mean() - 1.0) < 0.1 / np.sqrt(3 * x.size) * 5, name
        else:  # matrix: N(0, 0.02)
            assert abs(x.std() / 0.02 - 1) < 0.01, name
            assert abs(x.mean()) < 5 * 0.02 / np.sqrt(x.size), name


def test_same_seed_same_bytes_and_independent_tensors():
    a = synth.make_layer(QWEN3_0P6B, seed=7, layer=2)
    b = synth.make_layer(QWEN3_0P6B, seed=7, layer=2)
    c = synth.make_layer(QWEN3_0P6B, seed=8, layer=2)
    d = synth.make_layer(QWEN3_0P6B, seed=7, layer=3)
    for name in a:
        assert torch.equal(a[name], b[name]), name
        assert not torch.equal(a[name], c[name]), name
        assert not torch.equal(a[name], d[name]), name
    # the q and k projections of one layer are drawn from different streams
    assert not torch.equal(a["k_proj"], a["v_proj"])


def test_whole_model_and_a_subset_agree():
    cfg = dict(QWEN3_0P6B, n_layers=3, vocab=512)
    full = synth.make_weights(cfg, seed=2)
    part = synth.make_weights(cfg, seed=2, layers=[1])
    assert part["q_proj"][0] is None and part["q_proj"][2] is None
    for name in synth.LAYER_NAMES:
        assert torch.equal(full[name][1], part[name][1]), name
    assert full["lm_head"] is None  # tied embeddings: the head is the embedding matrix
    assert abs(_f(full["embed"]).std() / 0.02 - 1) < 0.02


def test_token_ids_uniform_and_seeded():
    V = 151936
    ids = synth.make_ids(V, 4, 50_000, seed=3)
    assert ids.dtype == torch.int32 and tuple(ids.shape) == (4, 50_000)
    x = ids.numpy().ravel()
    assert x.min() >= 0 and x.max() < V
    counts = np.bincount(x * 10 // V, minlength=10)  # ten equal bins of the vocabulary
    expected = x.size / 10
    assert np.all(np.abs(counts - expected) < 5 * np.sqrt(expected))
    assert torch.equal(ids, synth.make_ids(V, 4, 50_000, seed=3))
    assert not torch.equal(ids, synth.make_ids(V, 4, 50_000, seed=4))


def test_prefilled_kv_is_standard_normal():
    k = synth.make_kv_normal((2, 8, 4096, 128), seed=4, layer=0, which="k")
    v = synth.make_kv_normal((2, 8, 4096, 128), seed=4, layer=0, which="v")
    assert k.dtype == torch.bfloat16
    for t in (k, v):
        x = _f(t)
        assert abs(x.std() - 1) < 0.01 and abs(x.mean()) < 0.01
    assert not torch.equal(k, v)


def test_bit_round_trip():
    t = synth.make_layer(QWEN3_0P6B, seed=1, layer=0)["q_norm"]
    assert torch.equal(synth.from_numpy_bits(synth.to_numpy_bits(t)), t)
