"""Full-size parity of the generation features on sampled outputs, in the configurations
`bench.py --feature padded|prefix|window` times (Qwen3-0.6B shape for padding and prefix caching,
Qwen3-8B shape for the sliding window with a rolling buffer).

As in tests/test_gpu_fullsize.py, each checked layer is verified row by row from the GPU's own
tapped layer input and KV cache: the oracle recomputes q/k/v of sampled rows (the cache slots must
match, relative L2 <= 1e-3) and the attention + o_proj + MLP of those rows over the GPU cache with the
mask the pages' generation recipe gives them (layer output <= 1e-2); logits of the last rows <= 2e-2.
"""
import numpy as np
import pytest
import torch

from oracle import generation as G
from qwen3_decoder_transformer_gb300 import QWEN3_0P6B, QWEN3_8B, build as Bld, synth
from tests.test_gpu_fullsize import _host_layer
from tests.util import bits, rel_l2, top1_agreement, widen

pytestmark = pytest.mark.gpu
PAD = 151643 % QWEN3_0P6B["vocab"]


@pytest.fixture(scope="module")
def bd():
    Bld.build()
    from qwen3_decoder_transformer_gb300 import binding
    binding.lib()
    return binding


def _check_rows(om, layer, xin, xout, rows, pos, seqs, slots, kc_of, vc_of, masks):
    """rows: indices into xin/xout; seqs/slots: each row's sequence and cache slot; kc_of(b)/vc_of(b):
    the [Hkv, cap, dh] cache of sequence b as the kernels read it; masks[i]: visible slots of row i."""
    q, k, v = om.layer_qkv(layer, xin[rows], np.asarray(pos, np.int32))
    kg = np.stack([kc_of(b)[:, s] for b, s in zip(seqs, slots)])
    vg = np.stack([vc_of(b)[:, s] for b, s in zip(seqs, slots)])
    assert rel_l2(widen(kg), widen(k)) <= 1e-3 and rel_l2(widen(vg), widen(v)) <= 1e-3, layer
    sets = sorted(set(seqs))
    kc = np.stack([kc_of(b) for b in sets])
    vc = np.stack([vc_of(b) for b in sets])
    kvset = np.array([sets.index(b) for b in seqs], np.int32)
    out = om.layer_out_masked(layer, xin[rows], q, kc, vc, kvset, np.stack(masks))
    e = rel_l2(widen(xout[rows]), widen(out))
    assert e <= 1e-2, (layer, e)
    return out


def _padded_setup(seed, B, T, lo):
    rng = np.random.default_rng(seed)
    real = rng.integers(lo, T + 1, size=B)
    return real


def test_padded_batch_0p6b(bd):
    """32 prompts of 512..2048 tokens left-padded to 2048 (the padded-batch bench workload)."""
    cfg, seed, B, T = QWEN3_0P6B, 5, 32, 2048
    L, d, V = cfg["n_layers"], cfg["hidden"], cfg["vocab"]
    real = _padded_setup(seed, B, T, 512)
    w = synth.make_weights(cfg, seed, device="cuda")
    ids = synth.make_ids(V, B, T, seed, device="cuda")
    for b in range(B):
        ids[b, :T - int(real[b])] = PAD
    ids_h = ids.cpu().numpy()
    prompts = [list(ids_h[b, T - int(real[b]):]) for b in range(B)]
    _, _, positions, mask = G.left_pad(prompts, PAD, width=T)
    m = bd.Model(cfg, w, max_batch=B, capacity=T, max_tokens=B * T)
    # sampled rows: the shortest and longest prompt, one more; first real token, last token, a pad row
    order = np.argsort(real)
    seqs_pick = [int(order[0]), int(order[-1]), int(order[B // 2])]
    rows, seqs, slots = [], [], []
    for b in seqs_pick:
        first = T - int(real[b])
        cand = [first, T - 1, (first + T) // 2] + ([first - 1, 0] if first > 0 else [])
        for t in sorted(set(cand)):
            rows.append(b * T + t)
            seqs.append(b)
            slots.append(t)
    rows = np.array(rows)
    logits = torch.empty(B, V, dtype=torch.float32, device="cuda")
    for layer in (0, L - 1):
        xin = torch.empty(B * T, d, dtype=torch.bfloat16, device="cuda")
        xout = torch.empty_like(xin)
        m.set_length(0, 0)
        m.set_tap(layer, xin, xout)
        m.prefill_padded(ids, real, logits)
        assert m.get_error() == 0
        m.set_tap(-1)
        om = _host_layer(w, cfg, layer)
        k_gpu, v_gpu = m.kv_view(layer)
        cache = {b: (bits(k_gpu[b]), bits(v_gpu[b])) for b in set(seqs)}
        masks = [mask[b, t] for b, t in zip(seqs, slots)]
        pos = [positions[b, t] for b, t in zip(seqs, slots)]
        xo = bits(xout)
        _check_rows(om, layer, bits(xin), xo, rows, pos, seqs, slots, lambda b: cache[b][0],
                    lambda b: cache[b][1], masks)
    last = np.arange(B) * T + T - 1
    ref = om.head(xo[last])
    got = logits.cpu().numpy()
    assert rel_l2(got, ref) <= 2e-2
    assert top1_agreement(got, ref)[1] >= 0.99
    m.close()


@pytest.mark.parametrize("P", [2048, 2000], ids=["prefix2048", "prefix2000"])
def test_shared_prefix_0p6b(bd, P):
    """A P-token start shared by 32 prompts of 64..256 tokens (the prefix-caching bench workload;
    2000 leaves a partial 128-slot tile that is copied rather than shared)."""
    cfg, seed, B = QWEN3_0P6B, 6, 32
    L, d, V = cfg["n_layers"], cfg["hidden"], cfg["vocab"]
    rng = np.random.default_rng(seed)
    lens = rng.integers(64, 257, size=B)
    Tp = int(lens.max())
    w = synth.make_weights(cfg, seed, device="cuda")
    pre = synth.make_ids(V, 1, P, seed, device="cuda")
    body = synth.make_ids(V, B, Tp, seed + 1, device="cuda")
    for b in range(B):
        body[b, :Tp - int(lens[b])] = PAD
    body_h = body.cpu().numpy()
    prompts = [list(body_h[b, Tp - int(lens[b]):]) for b in range(B)]
    _, _, positions, mask = G.left_pad(prompts, PAD, start=P, width=Tp)
    cap = P + Tp
    m = bd.Model(cfg, w, max_batch=B, capacity=cap, max_tokens=B * Tp + P)
    psh = P // 128 * 128
    b_pick = [0, int(np.argmin(lens)), int(np.argmax(lens)), B - 1]
    rows, seqs, slots = [], [], []
    for b in sorted(set(b_pick)):
        first = Tp - int(lens[b])
        for t in sorted(set([first, Tp - 1, (first + Tp) // 2] + ([first - 1] if first > 0 else []))):
            rows.append(b * Tp + t)
            seqs.append(b)
            slots.append(P + t)
    rows = np.array(rows)
    l1 = torch.empty(1, V, dtype=torch.float32, device="cuda")
    logits = torch.empty(B, V, dtype=torch.float32, device="cuda")
    for layer in (0, L - 1):
        xin = torch.empty(B * Tp, d, dtype=torch.bfloat16, device="cuda")
        xout = torch.empty_like(xin)
        m.set_length(0, 0)
        m.prefill(pre, l1)
        m.share_prefix(B)
        m.set_tap(layer, xin, xout)
        m.prefill_padded(body, lens, logits)
        assert m.get_error() == 0
        m.set_tap(-1)
        om = _host_layer(w, cfg, layer)
        k_gpu, v_gpu = m.kv_view(layer)
        k0, v0 = bits(k_gpu[0]), bits(v_gpu[0])
        own = {b: (bits(k_gpu[b]), bits(v_gpu[b])) for b in set(seqs)}
        # the partial tile of the start is copied into every sequence bit for bit
        for b in own:
            assert np.array_equal(own[b][0][:, psh:P], k0[:, psh:P]) and np.array_equal(own[b][1][:, psh:P], v0[:, psh:P])
        # what the kernels read: whole tiles of the start from sequence 0, the rest from the sequence
        kc_of = lambda b: np.concatenate([k0[:, :psh], own[b][0][:, psh:]], axis=1)
        vc_of = lambda b: np.concatenate([v0[:, :psh], own[b][1][:, psh:]], axis=1)
        masks = []
        for b, s in zip(seqs, slots):
            mk = np.zeros(cap, bool)
            mk[:P + Tp] = mask[b, s - P]
            masks.append(mk)
        pos = [positions[b, s - P] for b, s in zip(seqs, slots)]
        xo = bits(xout)
        _check_rows(om, layer, bits(xin), xo, rows, pos, seqs, slots, kc_of, vc_of, masks)
    last = np.arange(B) * Tp + Tp - 1
    ref = om.head(xo[last])
    got = logits.cpu().numpy()
    assert rel_l2(got, ref) <= 2e-2
    assert top1_agreement(got, ref)[1] >= 0.99
    m.close()


def test_window_rolling_decode_8b(bd):
    """Window 4096 with a rolling buffer: 16 sequences decode at position 32768 (the window bench
    workload); the ring holds bf16 N(0, 1) keys and values for the last 4352 slots."""
    W, Bd, ctx = 4096, 16, 32768
    cfg = dict(QWEN3_8B, sliding_window=W, rolling_cache=1)
    seed = 7
    L, d, V, Hkv, dh = cfg["n_layers"], cfg["hidden"], cfg["vocab"], cfg["n_kv_heads"], cfg["head_dim"]
    w = synth.make_weights(cfg, seed, device="cuda")
    m = bd.Model(cfg, w, max_batch=Bd, capacity=ctx + 72, max_tokens=128)
    R = m.kv_view(0)[0].shape[2]
    for layer in range(L):
        k, v = m.kv_view(layer)
        k.copy_(synth.make_kv_normal((Bd, Hkv, R, dh), seed, layer, "k", device="cuda"))
        v.copy_(synth.make_kv_normal((Bd, Hkv, R, dh), seed, layer, "v", device="cuda"))
    ids = synth.make_ids(V, Bd, 1, seed, device="cuda").reshape(Bd)
    logits = torch.empty(Bd, V, dtype=torch.float32, device="cuda")
    b_pick = [0, 7, Bd - 1]
    keep = [(ctx - W + 1 + i) % R for i in range(W)]  # ring rows of the visible positions, oldest first
    for layer in (0, L - 1):
        xin = torch.empty(Bd, d, dtype=torch.bfloat16, device="cuda")
        xout = torch.empty_like(xin)
        m.set_length(ctx, Bd)
        m.set_tap(layer, xin, xout)
        m.decode_step(ids, logits)
        assert m.get_error() == 0
        m.set_tap(-1)
        om = _host_layer(w, cfg, layer)
        k_gpu, v_gpu = m.kv_view(layer)
        ring = {b: (bits(k_gpu[b]), bits(v_gpu[b])) for b in b_pick}
        kc_of = lambda b: np.ascontiguousarray(ring[b][0][:, keep])
        vc_of = lambda b: np.ascontiguousarray(ring[b][1][:, keep])
        masks = [np.ones(W, bool) for _ in b_pick]
        # the new token is the newest of the W gathered slots
        xo = bits(xout)
        _check_rows(om, layer, bits(xin), xo, np.array(b_pick), [ctx] * len(b_pick), b_pick, [W - 1] * len(b_pick),
                    kc_of, vc_of, masks)
    ref = om.head(xo)
    got = logits.cpu().numpy()
    assert rel_l2(got, ref) <= 2e-2
    assert top1_agreement(got, ref)[1] >= 0.99
    # later steps keep the ring bounded and the results finite
    for _ in range(3):
        m.decode_step(ids, logits)
    assert m.get_error() == 0 and m.length() == (ctx + 4, Bd) and torch.isfinite(logits).all()
    m.close()
