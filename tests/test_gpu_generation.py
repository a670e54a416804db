"""Generation features through the C ABI against the oracle's generation semantics ("A modern
architecture: Qwen3": batched generation with left padding, section 7 sliding windows and rolling
buffers, section 8 prefix caching), plus the greedy-token kernel.

Tiny config throughout; the oracle runs every case in full. Decode steps are teacher-forced with the
oracle's own tokens. Bars as for the plain forward pass: logits relative L2 <= 2e-2 and top-1 agreement
>= 99% on margin-clear rows; the greedy kernel is bit-exact (same fp32 logits on both sides).
"""
import numpy as np
import pytest
import torch

import oracle as O
from oracle import generation as G
from qwen3_decoder_transformer_gb300 import TINY, build as Bld, synth
from tests.util import bits, max_rel_rows, rel_l2, top1_agreement, widen

pytestmark = pytest.mark.gpu
STOP = 7


@pytest.fixture(scope="module")
def bd():
    Bld.build()
    from qwen3_decoder_transformer_gb300 import binding
    binding.lib()
    return binding


@pytest.fixture(scope="module")
def tiny(bd):
    w_host = synth.make_weights(TINY, 0)
    w_dev = {k: ([t.cuda() for t in v] if isinstance(v, list) else (None if v is None else v.cuda()))
             for k, v in w_host.items()}
    return w_dev, O.Model(TINY, synth.weights_to_numpy(w_host))


def _prompts(lengths, seed):
    rng = np.random.default_rng(seed)
    return [list(rng.integers(8, TINY["vocab"], size=n)) for n in lengths]


def _check_logits(got, ref, what):
    e = rel_l2(got, ref)
    assert e <= 2e-2, (what, e)
    raw, filt, _ = top1_agreement(got, ref)
    assert filt >= 0.99, (what, raw, filt)


# ------------------------------------------------------------------------------- greedy kernel

def test_greedy_kernel(bd):
    rng = np.random.default_rng(5)
    B, V = 6, TINY["vocab"]
    lg = rng.standard_normal((B, V)).astype(np.float32)
    lg[1, [5, 900]] = 100.0            # tie: lowest index
    lg[2, [17, 3]] = np.nan            # NaN counts as the largest, first one wins
    lg[3, :] = -np.inf                 # nothing finite: index 0
    lg[4, V - 1] = 50.0                # last element
    t = torch.from_numpy(lg).cuda()
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    bd.op_greedy(t, nxt)
    assert nxt.cpu().numpy().tolist() == np.argmax(lg, axis=1).tolist()
    # stop handling, against the oracle's statement of the rule
    stop = int(np.argmax(lg[0]))
    done0 = np.array([0, 1, 0, 0, 0, 1], dtype=np.int32)
    done = torch.from_numpy(done0.copy()).cuda()
    bd.op_greedy(t, nxt, stop_id=stop, done=done)
    ref_next, ref_done = G.greedy(lg, done0.astype(bool), stop)
    assert nxt.cpu().numpy().tolist() == ref_next.tolist()
    assert done.cpu().numpy().astype(bool).tolist() == ref_done.tolist()
    # a strided view of wider rows
    wide = torch.from_numpy(np.concatenate([lg, lg[:, :8]], axis=1)).cuda()
    bd.op_greedy(wide[:, :V], nxt)
    assert nxt.cpu().numpy().tolist() == np.argmax(lg, axis=1).tolist()


@pytest.mark.parametrize("B", [1, 3, 16, 64])
def test_greedy_kernel_split_rows(bd, B):
    """Vocabulary-sized rows (151,936 logits) are split over several CTAs per row and merged by the last
    one: ties, NaN and maxima placed across segment boundaries, with the workspace (split rows) and without
    it (one CTA per row), twice in a row (the tickets must be left at zero)."""
    rng = np.random.default_rng(50 + B)
    V = 151936
    lg = rng.standard_normal((B, V)).astype(np.float32)
    lg[0, [70000, 9000, 150000]] = 7.0                # tie across segments: lowest index
    if B > 1:
        lg[1, [120001, 80000]] = np.nan               # NaN wins, first NaN
        lg[1, 5] = 1e30
    if B > 2:
        lg[2, :] = -np.inf                            # nothing finite: index 0
    if B > 3:
        lg[3, V - 1] = 99.0                           # the very last element
        lg[4, 0] = 99.0                               # the very first element
    t = torch.from_numpy(lg).cuda()
    ref = np.argmax(lg, axis=1).tolist()
    work = torch.zeros(max(1, bd.greedy_workspace(B) // 4), dtype=torch.int32, device="cuda")
    for w in (work, work, None):
        nxt = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        bd.op_greedy(t, nxt, work=w)
        assert nxt.cpu().numpy().tolist() == ref
    assert not work[:64].any()


# ------------------------------------------------------------------------------- left padding

def _run_padded(bd, w, prompts, steps_o, cap, prefix_ids=None):
    """GPU: (prefix, share,) padded prefill, then decode steps fed with the oracle's tokens."""
    B = len(prompts)
    ids = torch.from_numpy(steps_o[0]["ids"]).cuda()
    width = ids.shape[1]
    V = TINY["vocab"]
    m = bd.Model(TINY, w, max_batch=B, capacity=cap, max_tokens=max(B * width, len(prefix_ids or [])))
    if prefix_ids is not None:
        pl = torch.empty(1, V, dtype=torch.float32, device="cuda")
        m.prefill(torch.tensor([prefix_ids], dtype=torch.int32, device="cuda"), pl)
        m.share_prefix(B)
    lg = torch.empty(B, V, dtype=torch.float32, device="cuda")
    m.prefill_padded(ids, [len(p) for p in prompts], lg)
    got = [lg.cpu().numpy()]
    feed = torch.empty(B, dtype=torch.int32, device="cuda")
    for k in range(1, len(steps_o)):
        feed.copy_(torch.from_numpy(steps_o[k]["ids"][:, 0]))
        m.decode_step(feed, lg)
        got.append(lg.cpu().numpy())
    assert m.get_error() == 0
    return m, got


@pytest.mark.parametrize("lengths", [[5, 64, 37, 100], [128, 77, 1], [300, 40, 129], [512, 3, 260]],
                         ids=["width100", "width128", "width300", "width512"])
def test_padded_prefill_and_decode(bd, tiny, lengths):
    w, om = tiny
    prompts = _prompts(lengths, 40 + len(lengths))
    rows, steps_o = G.generate(om, prompts, 6, STOP, keep=True)
    width = max(lengths)
    m, got = _run_padded(bd, w, prompts, steps_o, cap=width + 8)
    for k, g in enumerate(got):
        _check_logits(g, steps_o[k]["logits"], ("step", k))
    # layer-0 cache, real and padding slots alike, against the oracle's
    kc_o, vc_o = steps_o[-1]["cache"]
    n = width + len(steps_o) - 1
    k, v = m.kv_view(0)
    assert rel_l2(widen(bits(k[:len(lengths), :, :n])), widen(kc_o[0, :, :, :n])) <= 1e-3
    assert rel_l2(widen(bits(v[:len(lengths), :, :n])), widen(vc_o[0, :, :, :n])) <= 1e-3
    m.close()


def test_padded_all_rows(bd, tiny):
    """Every row of a padded prefill, padding rows included (each sees only itself)."""
    w, om = tiny
    prompts = _prompts([9, 40, 23], 50)
    ids, real, pos, mask = G.left_pad(prompts, STOP)
    B, T = ids.shape
    kc, vc = om.new_cache(B, T)
    ref = om.forward_masked(kc, vc, ids, pos, np.arange(T, dtype=np.int32)[None], mask, all_rows=True)
    m = bd.Model(TINY, w, max_batch=B, capacity=T, max_tokens=B * T)
    lg = torch.empty(B * T, TINY["vocab"], dtype=torch.float32, device="cuda")
    m.prefill_padded(torch.from_numpy(ids).cuda(), [len(p) for p in prompts], lg, all_rows=True)
    _check_logits(lg.cpu().numpy(), ref, "all rows")
    m.close()


def test_padding_errors(bd, tiny):
    w, _ = tiny
    m = bd.Model(TINY, w, max_batch=2, capacity=64, max_tokens=128)
    ids = torch.full((2, 8), STOP, dtype=torch.int32, device="cuda")
    lg = torch.empty(2, TINY["vocab"], dtype=torch.float32, device="cuda")
    for bad in ([0, 8], [9, 8]):
        with pytest.raises(bd.Qwen3Error):
            m.prefill_padded(ids, bad, lg)
    m.prefill_padded(ids, [3, 8], lg)
    with pytest.raises(bd.Qwen3Error):  # a second padded block
        m.prefill_padded(ids, [3, 8], lg)
    m.prefill_padded(ids, [8, 8], lg)   # unpadded continuation is fine
    with pytest.raises(bd.Qwen3Error):  # sharing needs a single sequence
        m.share_prefix(2)
    m.set_length(0, 0)
    m.prefill_padded(ids, [2, 5], lg)   # the layout was cleared
    assert m.length() == (8, 2)
    m.close()


# ------------------------------------------------------------------------------- shared prefix

@pytest.mark.parametrize("plen", [150, 256], ids=["prefix150", "prefix256"])
def test_shared_prefix(bd, tiny, plen):
    w, om = tiny
    pre = _prompts([plen], 60)[0]
    prompts = _prompts([12, 30, 7], 61)
    prefix = G.make_prefix(om, pre)
    rows, steps_o = G.generate(om, prompts, 5, STOP, prefix=prefix)
    m, got = _run_padded(bd, w, prompts, steps_o, cap=plen + 40, prefix_ids=pre)
    for k, g in enumerate(got):
        _check_logits(g, steps_o[k]["logits"], ("step", k))
    m.close()


# ------------------------------------------------------------------------------- generate loop

def test_generate_loop(bd, tiny):
    w, om = tiny
    prompts = _prompts([11, 30, 4], 70)
    B, max_new = len(prompts), 6
    ids, real, _, _ = G.left_pad(prompts, STOP)
    m = bd.Model(TINY, w, max_batch=B, capacity=ids.shape[1] + max_new, max_tokens=B * ids.shape[1])
    out = torch.full((B, max_new), -1, dtype=torch.int32, device="cuda")
    steps = m.generate(torch.from_numpy(ids).cuda(), [len(p) for p in prompts], max_new, -1, out)
    assert steps == max_new
    toks = out.cpu().numpy()
    # each choice is the oracle's argmax given the same history, up to near-ties
    _, steps_o = G.generate(om, prompts, max_new, -1, forced=[toks[:, k] for k in range(max_new - 1)], pad_id=STOP)
    for k in range(max_new):
        ref = steps_o[k]["logits"]
        best = ref.max(axis=1)
        chosen = ref[np.arange(B), toks[:, k]]
        assert np.all(best - chosen <= 4e-2 * np.abs(ref).max()), k
    # stop id: a row that emits it keeps emitting it; the loop ends when all rows are done
    m.set_length(0, 0)
    stop = int(toks[0, 1])
    out.fill_(-1)
    steps = m.generate(torch.from_numpy(ids).cuda(), [len(p) for p in prompts], max_new, stop, out)
    got = out.cpu().numpy()[:, :steps]
    for r in got:
        hit = np.nonzero(r == stop)[0]
        if hit.size:
            assert np.all(r[hit[0]:] == stop)
    if steps < max_new:
        assert all((r == stop).any() for r in got)
    m.close()


# ------------------------------------------------------------------------------- sliding window

def _window_model(bd, w, W, rolling, B, cap, max_tokens):
    cfg = dict(TINY, sliding_window=W, rolling_cache=int(rolling))
    return bd.Model(cfg, w, max_batch=B, capacity=cap, max_tokens=max_tokens)


@pytest.mark.parametrize("rolling", [False, True], ids=["banded", "rolling"])
def test_sliding_window(bd, tiny, rolling):
    """Prefill in chunks (whole 128-row tiles and ragged ones), then decode steps; every row against the
    oracle's banded mask over the whole sequence. The rolling buffer wraps several times."""
    w, om = tiny
    W, B = 100, 2
    chunks = [128, 128, 37, 91, 60]
    n_dec = 6
    total = sum(chunks) + n_dec
    ids = synth.make_ids(TINY["vocab"], B, total, 80).numpy()
    V = TINY["vocab"]
    ref = np.stack([G.banded(om, ids[b], W) for b in range(B)])  # [B, total, V]
    m = _window_model(bd, w, W, rolling, B, cap=total, max_tokens=B * 128)
    if rolling:
        k, _ = m.kv_view(0)
        assert k.shape[2] == 256  # ring of W + 128 - 1 slots, rounded up to 256
    pos = 0
    for T in chunks:
        lg = torch.empty(B * T, V, dtype=torch.float32, device="cuda")
        m.prefill(torch.from_numpy(np.ascontiguousarray(ids[:, pos:pos + T])).cuda(), lg, all_rows=True)
        _check_logits(lg.cpu().numpy(), ref[:, pos:pos + T].reshape(B * T, V), ("chunk at", pos))
        pos += T
    feed = torch.empty(B, dtype=torch.int32, device="cuda")
    lg = torch.empty(B, V, dtype=torch.float32, device="cuda")
    for s in range(n_dec):
        feed.copy_(torch.from_numpy(ids[:, pos]))
        m.decode_step(feed, lg)
        _check_logits(lg.cpu().numpy(), ref[:, pos], ("decode at", pos))
        pos += 1
    assert m.get_error() == 0
    m.close()


def test_rolling_chunk_limit(bd, tiny):
    w, _ = tiny
    m = _window_model(bd, w, 100, True, 1, cap=1000, max_tokens=128)
    ids = torch.zeros(1, 158, dtype=torch.int32, device="cuda")  # > ring - window + 1 = 157
    lg = torch.empty(1, TINY["vocab"], dtype=torch.float32, device="cuda")
    with pytest.raises(bd.Qwen3Error):
        m.prefill(ids, lg)
    with pytest.raises(bd.Qwen3Error):  # padding is not combined with a window
        m.prefill_padded(ids[:, :8], [4], lg)
    m.close()


# ------------------------------------------------------------------------------- attention ops

def _rand(rng, shape):
    return synth.to_numpy_bits(torch.from_numpy(rng.standard_normal(shape)).to(torch.bfloat16))


@pytest.mark.parametrize("ps,psh,pads", [(300, 256, [0, 17, 250]), (0, 0, [0, 600, 512])])
def test_decode_attention_layout_op(bd, ps, psh, pads):
    """Decode attention with padding slots and a shared prefix, against masked oracle rows. In the second
    layout the first 512-slot chunk of rows 1 and 2 is padding only: its record has no visible key, and
    its output floats (NaN from the workspace's initial contents) must not reach the result."""
    rng = np.random.default_rng(90)
    B, Hq, Hkv, dh, cap = 3, 8, 2, 128, 1024
    n = 700  # query slot = 699 after the cache holds 700 slots
    q = _rand(rng, (B, Hq, dh))
    kc = _rand(rng, (B, Hkv, cap, dh))
    vc = _rand(rng, (B, Hkv, cap, dh))
    meta = np.array([ps, psh] + pads, dtype=np.int32)
    out = torch.empty(B, Hq * dh, dtype=torch.bfloat16, device="cuda")
    work = torch.full((bd.attention_decode_workspace(B, Hq, dh, cap) // 4 + 1,), float("nan"), dtype=torch.float32,
                      device="cuda")
    len_t = torch.tensor([n - 1], dtype=torch.int32, device="cuda")
    bd.op_attention_decode(synth.from_numpy_bits(q, "cuda"), synth.from_numpy_bits(kc, "cuda"),
                           synth.from_numpy_bits(vc, "cuda"), len_t, work, out,
                           seq_meta=torch.from_numpy(meta).cuda())
    got = widen(bits(out)).reshape(B, Hq, dh)
    for b in range(B):
        src_k = np.concatenate([kc[0, :, :psh], kc[b, :, psh:]], axis=1)
        src_v = np.concatenate([vc[0, :, :psh], vc[b, :, psh:]], axis=1)
        mask = np.zeros(cap, bool)
        mask[:n] = True
        mask[ps:ps + pads[b]] = False
        ref = O.attention_masked_gqa_row_f64(q[b], src_k, src_v, mask)
        assert np.isfinite(got[b]).all(), b
        assert rel_l2(got[b], ref) <= 1e-2, b
        assert max_rel_rows(got[b], ref, dh) <= 3e-2, b


@pytest.mark.parametrize("heads", [0, 2])
def test_prefill_attention_window_ring_op(bd, heads):
    """Prefill attention over a rolling buffer with a window, against oracle rows gathered by position,
    with the automatic kernel choice and with two heads per CTA."""
    rng = np.random.default_rng(91)
    B, Hq, Hkv, dh, T, W, R = 2, 8, 4, 64, 128, 100, 256
    len0 = 300  # positions 300..427 read keys back to 201, rows p mod 256
    q = _rand(rng, (B, Hq, T, dh))
    kc = _rand(rng, (B, Hkv, R, dh))
    vc = _rand(rng, (B, Hkv, R, dh))
    out = torch.empty(B * T, Hq * dh, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    len_t = torch.tensor([len0], dtype=torch.int32, device="cuda")
    bd.op_attention_prefill(synth.from_numpy_bits(q, "cuda"), synth.from_numpy_bits(kc, "cuda"),
                            synth.from_numpy_bits(vc, "cuda"), len_t, out, err=err, window=W, ring=R,
                            heads_per_cta=heads)
    assert int(err.item()) == 0
    got = widen(bits(out)).reshape(B, T, Hq, dh)
    for b in range(B):
        for t in (0, 1, 63, 64, 127):
            p = len0 + t
            keys = [(s % R) for s in range(p - W + 1, p + 1)]
            ref = O.attention_gqa_row_f64(q[b, :, t], np.ascontiguousarray(kc[b][:, keys]),
                                          np.ascontiguousarray(vc[b][:, keys]), W)
            assert rel_l2(got[b, t], ref) <= 1e-2, (b, t)


@pytest.mark.parametrize("heads,T", [(1, 300), (2, 300), (1, 4200), (1, 16500)])
def test_prefill_attention_padding_op(bd, heads, T):
    """Prefill attention with left padding at the start of the block (a padded prompt batch), one and two
    heads per CTA, against masked oracle rows: a real token sees the real slots up to its own, a padding
    slot sees only itself. Row 2's padding covers the first 128-slot tile whole (skipped by the kernels).
    At 4200 keys the persistent kernel takes its speculative form, where the rows of one warp reach their
    first visible key at different tiles; at 16500 keys its alternating form (two softmax warpgroups, used from
    8192 keys)."""
    rng = np.random.default_rng(92)
    B, Hq, Hkv, dh = 3, 8, 2, 128
    pads = [0, 37, 200]
    q = _rand(rng, (B, Hq, T, dh))
    kc = _rand(rng, (B, Hkv, T, dh))
    vc = _rand(rng, (B, Hkv, T, dh))
    meta = torch.tensor([0, 0] + pads, dtype=torch.int32, device="cuda")
    out = torch.empty(B * T, Hq * dh, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    len_t = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.op_attention_prefill(synth.from_numpy_bits(q, "cuda"), synth.from_numpy_bits(kc, "cuda"),
                            synth.from_numpy_bits(vc, "cuda"), len_t, out, err=err, seq_meta=meta,
                            heads_per_cta=heads)
    assert int(err.item()) == 0
    got = widen(bits(out)).reshape(B, T, Hq, dh)
    for b in range(B):
        for t in sorted({0, 5, 36, 37, 127, 128, 199, 200, 201, 255, 256, T - 1}):
            mask = np.zeros(T, bool)
            mask[:t + 1] = True
            mask[:pads[b]] = False
            mask[t] = True
            ref = O.attention_masked_gqa_row_f64(q[b, :, t], kc[b], vc[b], mask)
            assert np.isfinite(got[b, t]).all(), (b, t)
            assert rel_l2(got[b, t], ref) <= 1e-2, (b, t)
            assert max_rel_rows(got[b, t], ref, dh) <= 3e-2, (b, t)
