"""Model-level pins for the oracle: invariants the pages' cache contract fixes (cached decode equals
the uncached forward, causal prefix, batch independence, KV-cache slot = position), and agreement
with an fp64 PyTorch statement of the model to within bf16 rounding noise."""
import numpy as np
import pytest

import oracle as O
from qwen3_decoder_transformer_gb300 import TINY, synth
from tests.model_f64 import forward_f64

CFG = TINY


@pytest.fixture(scope="module")
def tiny():
    w = synth.make_weights(CFG, 0)
    return w, O.Model(CFG, synth.weights_to_numpy(w))


def check_cached_equals_uncached(m):
    ids = synth.make_ids(CFG["vocab"], 1, 20, 7).numpy()
    kc, vc = m.new_cache(1, 32)
    full = m.forward(kc, vc, ids, 0)
    kc2, vc2 = m.new_cache(1, 32)
    m.forward(kc2, vc2, ids[:, :19], 0)
    step = m.forward(kc2, vc2, ids[:, 19:], 19)
    assert np.array_equal(full, step)
    assert np.array_equal(kc, kc2) and np.array_equal(vc, vc2)


def check_causal_prefix(m):
    ids = synth.make_ids(CFG["vocab"], 1, 24, 8).numpy()
    kc, vc = m.new_cache(1, 32)
    full = m.forward(kc, vc, ids, 0, all_rows=True)
    kc, vc = m.new_cache(1, 32)
    part = m.forward(kc, vc, ids[:, :10], 0, all_rows=True)
    assert np.array_equal(full[:10], part)


def check_batch_independence(m):
    ids = synth.make_ids(CFG["vocab"], 2, 12, 9).numpy()
    kc, vc = m.new_cache(2, 16)
    both = m.forward(kc, vc, ids, 0)
    for b in range(2):
        k1, v1 = m.new_cache(1, 16)
        one = m.forward(k1, v1, ids[b:b + 1], 0)
        assert np.array_equal(both[b], one[0])
        assert np.array_equal(kc[:, b], k1[:, 0])


def check_cache_slots(m):
    """Slot (l, b, j, p) of the cache holds layer l's k/v of sequence b, kv head j, position p."""
    ids = synth.make_ids(CFG["vocab"], 2, 6, 10).numpy()
    cap = 8
    kc, vc = m.new_cache(2, cap)
    _, tin, _ = m.forward(kc, vc, ids, 0, tap_layer=1)
    pos = np.tile(np.arange(6, dtype=np.int32), 2)
    q, k, v = m.layer_qkv(1, tin, pos)
    L, B, H, C, D = kc.shape
    flat_k, flat_v = kc.ravel(), vc.ravel()
    for r in range(12):
        b, p = divmod(r, 6)
        for j in range(H):
            addr = (((1 * B + b) * H + j) * C + p) * D  # closed form of the [L][B][Hkv][cap][dh] layout
            assert np.array_equal(flat_k[addr:addr + D], k[r, j])
            assert np.array_equal(flat_v[addr:addr + D], v[r, j])
    assert not kc[:, :, :, 6:].any()  # slots past the written positions stay untouched


def check_matches_f64_statement(w, m):
    ids = synth.make_ids(CFG["vocab"], 2, 48, 0)
    ref = forward_f64(CFG, w, ids).numpy()
    kc, vc = m.new_cache(2, 64)
    got = m.forward(kc, vc, ids.numpy(), 0, all_rows=True)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    # bf16 rounding noise is ~1e-2 here; every structural mistake tried gives > 0.1
    assert rel < 3e-2, rel


def check_errors(m):
    kc, vc = m.new_cache(1, 8)
    with pytest.raises(ValueError):
        m.forward(kc, vc, np.array([[CFG["vocab"]]], dtype=np.int32), 0)
    with pytest.raises(ValueError):
        m.forward(kc, vc, np.zeros((1, 9), dtype=np.int32), 0)


def test_cached_equals_uncached(tiny):
    check_cached_equals_uncached(tiny[1])


def test_causal_prefix(tiny):
    check_causal_prefix(tiny[1])


def test_batch_independence(tiny):
    check_batch_independence(tiny[1])


def test_cache_slots(tiny):
    check_cache_slots(tiny[1])


def test_matches_f64_statement(tiny):
    check_matches_f64_statement(*tiny)


def test_errors(tiny):
    check_errors(tiny[1])
