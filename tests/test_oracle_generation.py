"""Pins for the oracle's general (masked) forward pass and the generation semantics built on it:
left padding, shared prefixes, sliding windows and rolling buffers ("A modern architecture: Qwen3",
the batched-generation section, section 7 on sliding-window attention and section 8 on prefix
caching). Each check compares two routes the pages say must agree, or reduces to the pinned
equal-length forward pass."""
import numpy as np
import pytest

import oracle as O
from oracle import generation as G
from qwen3_decoder_transformer_gb300 import TINY, synth
from tests.util import rel_l2

CFG = TINY
STOP = 7  # a token id used as padding and stop id


def _model():
    return O.Model(CFG, synth.weights_to_numpy(synth.make_weights(CFG, 0)))


def _prompts(lengths, seed):
    rng = np.random.default_rng(seed)
    return [list(rng.integers(8, CFG["vocab"], size=n)) for n in lengths]


def check_masked_reduces_to_forward(m=None):
    """Causal mask, slot = position = column: the general forward equals the equal-length forward
    bit for bit (prefill of 2 x 12 tokens, then three decode steps)."""
    m = m or _model()
    ids = synth.make_ids(CFG["vocab"], 2, 15, 21).numpy()
    cap = 16
    ka, va = m.new_cache(2, cap)
    kb, vb = m.new_cache(2, cap)
    t = np.arange(12)
    mask = np.zeros((2, 12, cap), bool)
    mask[:, :, :12] = t[None, :] <= t[:, None]
    a = m.forward(ka, va, ids[:, :12], 0, all_rows=True)
    b = m.forward_masked(kb, vb, ids[:, :12], t[None], t[None], mask, all_rows=True)
    assert np.array_equal(a, b)
    for p in range(12, 15):
        a = m.forward(ka, va, ids[:, p:p + 1], p)
        mk = np.zeros((2, 1, cap), bool)
        mk[:, :, :p + 1] = True
        b = m.forward_masked(kb, vb, ids[:, p:p + 1], np.int32(p), np.int32(p), mk)
        assert np.array_equal(a, b)
    assert np.array_equal(ka, kb) and np.array_equal(va, vb)


def check_padding_invariance(m=None):
    """Padding gets no attention and positions count from the first real token: each row of a
    left-padded batch generates exactly what it generates alone, logits bit for bit."""
    m = m or _model()
    prompts = _prompts([5, 11, 8], 22)
    rows, steps = G.generate(m, prompts, 4, STOP)
    for b, p in enumerate(prompts):
        r1, s1 = G.generate(m, [p], 4, STOP)
        assert rows[b] == r1[0]
        for k in range(len(s1)):
            assert np.array_equal(steps[k]["logits"][b], s1[k]["logits"][0]), (b, k)


def check_pad_rows_see_themselves(m=None):
    """Without a prefix a padding token sees only itself (all padding shares id and position 0), so
    every padding row's output equals a lone pad token's at position 0."""
    m = m or _model()
    prompts = _prompts([3, 9], 23)
    ids, real, pos, mask = G.left_pad(prompts, STOP)
    B, T = ids.shape
    kc, vc = m.new_cache(B, T)
    logits = m.forward_masked(kc, vc, ids, pos, np.arange(T, dtype=np.int32)[None], mask, all_rows=True)
    k1, v1 = m.new_cache(1, 1)
    lone = m.forward(k1, v1, np.array([[STOP]], np.int32), 0)
    n_pad = T - len(prompts[0])
    assert n_pad > 1 and np.all(pos[0, :n_pad] == 0) and pos[0, n_pad] == 0 and pos[0, -1] == len(prompts[0]) - 1
    for t in range(n_pad):
        assert np.array_equal(logits[t], lone[0])


def check_prefix_equals_concatenation(m=None):
    """A shared prefix computed once (section 8) gives, row by row, what the concatenated prompt
    gives alone: same tokens and logits bit for bit, padding included."""
    m = m or _model()
    pre = _prompts([6], 24)[0]
    prompts = _prompts([4, 7], 25)
    prefix = G.make_prefix(m, pre)
    rows, steps = G.generate(m, prompts, 3, STOP, prefix=prefix)
    for b, p in enumerate(prompts):
        r1, s1 = G.generate(m, [pre + p], 3, STOP)
        assert rows[b] == r1[0]
        for k in range(len(s1)):
            assert np.array_equal(steps[k]["logits"][b], s1[k]["logits"][0]), (b, k)


def check_band_equals_rolling(m=None):
    """Section 7's experiment (34 tokens, window 16): the banded mask over a full cache and a rolling
    buffer of 16 slots, token by token with no mask, agree (to fp64 summation order)."""
    m = m or _model()
    ids = synth.make_ids(CFG["vocab"], 1, 34, 26).numpy()
    a = G.banded(m, ids, 16)
    b = G.rolling_stepwise(m, ids, 16)
    assert a.shape == b.shape == (34, CFG["vocab"])
    assert rel_l2(b, a) <= 1e-6
    # the window is real: a full causal pass differs beyond the window
    c = G.banded(m, ids, 34)
    assert np.array_equal(a[:16], c[:16]) and rel_l2(a[16:], c[16:]) > 1e-3


def check_window_limits(m=None):
    """W >= T is plain causal attention (bit for bit); W = 1 lets each token see only itself, so row i
    equals that token alone at position i."""
    m = m or _model()
    ids = synth.make_ids(CFG["vocab"], 1, 10, 27).numpy()
    kc, vc = m.new_cache(1, 10)
    causal = m.forward(kc, vc, ids, 0, all_rows=True)
    assert np.array_equal(G.banded(m, ids, 10), causal)
    one = G.banded(m, ids, 1)
    for i in (0, 4, 9):
        k1, v1 = m.new_cache(1, 16)
        mk = np.zeros((1, 1, 16), bool)
        mk[0, 0, 3] = True
        alone = m.forward_masked(k1, v1, ids[:, i:i + 1], np.int32(i), np.int32(3), mk)
        assert np.array_equal(one[i], alone[0])


def check_stop_semantics(m=None):
    """A finished row keeps emitting the stop id and is cut at its first stop id; generation ends
    when every row has finished."""
    m = m or _model()
    prompts = _prompts([4, 6], 28)
    _, steps = G.generate(m, prompts, 1, STOP)
    first = np.argmax(steps[0]["logits"], axis=1)
    stop = int(first[0])  # row 0 stops at once
    rows, steps = G.generate(m, prompts, 5, stop)
    assert rows[0] == []
    assert 1 <= len(steps) <= 5
    rows2, steps2 = G.generate(m, prompts[:1], 5, stop)
    assert rows2 == [[]] and len(steps2) == 1  # everyone finished after the first token


ALL_CHECKS = [check_masked_reduces_to_forward, check_padding_invariance, check_pad_rows_see_themselves,
              check_prefix_equals_concatenation, check_band_equals_rolling, check_window_limits,
              check_stop_semantics]


@pytest.fixture(scope="module")
def model():
    return _model()


@pytest.mark.parametrize("chk", ALL_CHECKS, ids=[c.__name__ for c in ALL_CHECKS])
def test_generation_pin(chk, model):
    chk(model)


def test_left_pad_recipe():
    """The padding recipe on a hand-checked case: prompts [a b] and [c d e] after a 2-slot prefix."""
    ids, real, pos, mask = G.left_pad([[11, 12], [13, 14, 15]], 0, start=2)
    assert ids.tolist() == [[0, 11, 12], [13, 14, 15]]
    assert real.tolist() == [[1, 1, 0, 1, 1], [1, 1, 1, 1, 1]]
    assert pos.tolist() == [[1, 2, 3], [2, 3, 4]]  # the pad sits at the prefix's last position
    assert mask[0].astype(int).tolist() == [[1, 1, 1, 0, 0], [1, 1, 0, 1, 0], [1, 1, 0, 1, 1]]
    assert mask[1].astype(int).tolist() == [[1, 1, 1, 0, 0], [1, 1, 1, 1, 0], [1, 1, 1, 1, 1]]


def test_masked_row_errors(model):
    q = np.zeros((CFG["n_q_heads"], CFG["head_dim"]), np.uint16)
    kc = np.zeros((CFG["n_kv_heads"], 4, CFG["head_dim"]), np.uint16)
    with pytest.raises(ValueError):
        O.attention_masked_gqa_row_f64(q, kc, kc, np.zeros(4, bool))
    kc2, vc2 = model.new_cache(1, 4)
    with pytest.raises(ValueError):
        model.forward_masked(kc2, vc2, np.array([[1]], np.int32), np.int32(0), np.int32(4), np.ones((1, 1, 4), bool))
