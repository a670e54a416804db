"""Whole-model parity through the C ABI (qwen3_init / qwen3_prefill / qwen3_decode_step).

Tiny config: the oracle runs the whole thing (prefill of 64 tokens + 8 greedy decode steps). Decode is
teacher-forced with the oracle's own greedy tokens so that one near-tie cannot cascade. Bars: per-layer
output relative L2 <= 1e-2, logits <= 2e-2, top-1 agreement >= 99% (raw, and on rows whose oracle
top-1/top-2 margin exceeds 4x the largest logit error).
"""
import numpy as np
import pytest
import torch

import oracle as O
from qwen3_decoder_transformer_gb300 import TINY, build as Bld, synth
from tests.util import bits, rel_l2, top1_agreement, widen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bd():
    Bld.build()
    from qwen3_decoder_transformer_gb300 import binding
    binding.lib()
    return binding


@pytest.fixture(scope="module")
def tiny(bd):
    cfg = TINY
    w_host = synth.make_weights(cfg, 0)
    w_dev = {k: ([t.cuda() for t in v] if isinstance(v, list) else (None if v is None else v.cuda()))
             for k, v in w_host.items()}
    om = O.Model(cfg, synth.weights_to_numpy(w_host))
    return cfg, w_dev, om


def test_tiny_prefill_and_decode(bd, tiny):
    cfg, w, om = tiny
    T, steps, cap = 64, 8, 80
    V, d, L = cfg["vocab"], cfg["hidden"], cfg["n_layers"]
    ids = synth.make_ids(V, 1, T, 0)
    m = bd.Model(cfg, w, max_batch=1, capacity=cap, max_tokens=T)
    logits = torch.empty(T, V, dtype=torch.float32, device="cuda")
    taps = {}
    for layer in range(L):
        taps[layer] = (torch.empty(T, d, dtype=torch.bfloat16, device="cuda"),
                       torch.empty(T, d, dtype=torch.bfloat16, device="cuda"))
    # one prefill per tapped layer would change the cache; tap layer 0 and L-1 on two contexts
    m.set_tap(L - 1, *taps[L - 1])
    m.prefill(ids.cuda(), logits, all_rows=True)
    assert m.get_error() == 0
    kc_o, vc_o = om.new_cache(1, cap)
    ref, tin, tout = om.forward(kc_o, vc_o, ids.numpy(), 0, all_rows=True, tap_layer=L - 1)
    got = logits.cpu().numpy()
    assert rel_l2(widen(bits(taps[L - 1][0])), widen(tin)) <= 1e-2
    assert rel_l2(widen(bits(taps[L - 1][1])), widen(tout)) <= 1e-2
    assert rel_l2(got, ref) <= 2e-2, rel_l2(got, ref)
    raw, filt, n = top1_agreement(got, ref)
    assert filt >= 0.99 and raw >= 0.95, (raw, filt, n)
    # KV cache: layer 0 keys depend only on the embedding rows and layer-0 weights
    for layer in range(L):
        k, v = m.kv_view(layer)
        tol = 1e-3 if layer == 0 else 1e-2
        assert rel_l2(widen(bits(k[0, :, :T])), widen(kc_o[layer, 0, :, :T])) <= tol
        assert rel_l2(widen(bits(v[0, :, :T])), widen(vc_o[layer, 0, :, :T])) <= tol
        assert not bits(k[0, :, T:]).any()
    assert m.length() == (T, 1)
    # greedy decode, teacher-forced with the oracle's tokens
    m.set_tap(-1)
    tok = int(ref[-1].argmax())
    step_logits = torch.empty(1, V, dtype=torch.float32, device="cuda")
    ids_dev = torch.empty(1, dtype=torch.int32, device="cuda")
    agree = []
    for s in range(steps):
        ids_dev.fill_(tok)
        m.decode_step(ids_dev, step_logits)
        r = om.forward(kc_o, vc_o, np.array([[tok]], dtype=np.int32), T + s)
        g = step_logits.cpu().numpy()
        assert rel_l2(g, r) <= 2e-2, (s, rel_l2(g, r))
        agree.append(int(g.argmax()) == int(r.argmax()))
        tok = int(r.argmax())
    assert m.get_error() == 0
    assert m.length() == (T + steps, 1)
    assert sum(agree) >= steps - 1
    m.close()


def test_tiny_errors(bd, tiny):
    cfg, w, _ = tiny
    V = cfg["vocab"]
    m = bd.Model(cfg, w, max_batch=2, capacity=16, max_tokens=32)
    logits = torch.empty(2, V, dtype=torch.float32, device="cuda")
    with pytest.raises(bd.Qwen3Error) as e:
        m.prefill(torch.zeros(1, 17, dtype=torch.int32, device="cuda"), logits)
    assert e.value.code == 3  # overflow: 17 > capacity 16
    with pytest.raises(bd.Qwen3Error) as e:
        m.prefill(torch.zeros(3, 4, dtype=torch.int32, device="cuda"), logits)
    assert e.value.code == 4  # batch above max_batch
    bad = torch.tensor([[1, V + 5]], dtype=torch.int32, device="cuda")
    m.prefill(bad, logits)
    assert m.get_error() == 7  # token id out of range, reported by the device flag
    assert m.get_error() == 0  # flag cleared
    with pytest.raises(bd.Qwen3Error) as e:
        bd.Model(dict(cfg, max_positions=8), w, max_batch=1, capacity=16)
    assert e.value.code == 2  # capacity above max_positions
    m.close()


def test_tiny_chunked_prefill_long_context(bd, tiny):
    """A short prefill chunk after a long context: the attention splits each query tile's key range
    over several CTAs (the runtime's split plan) and merges them; logits and the new cache rows must
    match the oracle running the same two calls."""
    cfg, w, om = tiny
    V = cfg["vocab"]
    T0, T1, cap = 1024, 64, 1100
    ids = synth.make_ids(V, 1, T0 + T1, 11)
    m = bd.Model(cfg, w, max_batch=1, capacity=cap, max_tokens=T0)
    logits = torch.empty(1, V, dtype=torch.float32, device="cuda")
    m.prefill(ids[:, :T0].cuda().contiguous(), logits)
    m.prefill(ids[:, T0:].cuda().contiguous(), logits)
    assert m.get_error() == 0
    kc, vc = om.new_cache(1, cap)
    om.forward(kc, vc, ids[:, :T0].numpy(), 0)
    ref = om.forward(kc, vc, ids[:, T0:].numpy(), T0)
    got = logits.cpu().numpy()
    assert rel_l2(got, ref) <= 2e-2
    k, v = m.kv_view(cfg["n_layers"] - 1)
    assert rel_l2(widen(bits(k[0, :, T0:T0 + T1])), widen(kc[-1, 0, :, T0:T0 + T1])) <= 1e-2
    m.close()


def test_tiny_graph_replay_matches_eager(bd, tiny):
    """Repeated forward calls replay a captured CUDA graph: the replay equals the eager pass bit for bit,
    reads the current contents of the id buffer, follows the cache length, and stays correct after the
    graph cache has dropped entries (more distinct calls than it keeps)."""
    cfg, w, _ = tiny
    V = cfg["vocab"]
    T, cap = 32, 256
    m = bd.Model(cfg, w, max_batch=1, capacity=cap, max_tokens=T)
    ids = synth.make_ids(V, 1, T, 3).cuda()
    logits = torch.empty(1, V, dtype=torch.float32, device="cuda")

    def run(eager, fn):
        m.set_timing(eager)  # timing runs the pass eagerly
        m.set_length(0, 0)
        fn()
        torch.cuda.synchronize()
        m.set_timing(False)
        return logits.clone()

    pre = lambda: m.prefill(ids, logits)
    ref = run(True, pre)
    assert torch.equal(run(False, pre), ref)  # capture + launch
    assert torch.equal(run(False, pre), ref)  # replay
    ids.copy_(synth.make_ids(V, 1, T, 4).cuda())  # same buffer, new contents
    ref2 = run(True, pre)
    assert not torch.equal(ref2, ref)
    assert torch.equal(run(False, pre), ref2)

    # decode steps after the prefill: graph replays against the eager steps
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")

    def steps(eager, n):
        out = []
        m.set_timing(eager)
        m.set_length(0, 0)
        m.prefill(ids, logits)
        for k in range(n):
            tok.fill_(k + 1)
            m.decode_step(tok, logits)
            out.append(logits.clone())
        torch.cuda.synchronize()
        m.set_timing(False)
        return out

    assert all(torch.equal(a, b) for a, b in zip(steps(False, 4), steps(True, 4)))

    # more distinct prefill calls than the graph cache keeps, then the first one again
    outs = {}
    for t in range(4, 4 + 20):
        part = ids[:, :t].contiguous()
        outs[t] = run(False, lambda: m.prefill(part, logits))
    for t in (4, 23):
        part = ids[:, :t].contiguous()
        assert torch.equal(run(True, lambda: m.prefill(part, logits)), outs[t])
    assert m.get_error() == 0
    m.close()


def test_tiny_decode_roomy_capacity_across_chunks(bd, tiny):
    """Decode with a capacity far above the length (4096 slots for about 512 tokens): the decode-attention
    grid covers only the 512-slot context chunks that hold keys, and the captured decode graph is swapped
    when the length crosses a chunk boundary (slot 511 -> 512 during these steps). Cache slots past the
    length hold NaN, which must never be read. Teacher-forced against the oracle, and the graph replays
    equal the eager steps bit for bit."""
    cfg, w, om = tiny
    V = cfg["vocab"]
    T, steps, cap = 508, 8, 4096
    ids = synth.make_ids(V, 1, T, 12)
    kc_o, vc_o = om.new_cache(1, cap)
    ref = om.forward(kc_o, vc_o, ids.numpy(), 0)
    toks = [int(ref[-1].argmax())]
    refs = []
    for s in range(steps):
        r = om.forward(kc_o, vc_o, np.array([[toks[-1]]], dtype=np.int32), T + s)
        refs.append(r)
        toks.append(int(r.argmax()))

    m = bd.Model(cfg, w, max_batch=1, capacity=cap, max_tokens=T)
    logits = torch.empty(1, V, dtype=torch.float32, device="cuda")
    ids_dev = torch.empty(1, dtype=torch.int32, device="cuda")

    def run(eager):
        m.set_timing(eager)
        m.set_length(0, 0)
        for layer in range(cfg["n_layers"]):  # stale slots past the length: NaN
            k, v = m.kv_view(layer)
            k.view(torch.int16).fill_(0x7FC0)
            v.view(torch.int16).fill_(0x7FC0)
        m.prefill(ids.cuda(), logits)
        out = []
        for s in range(steps):
            ids_dev.fill_(toks[s])
            m.decode_step(ids_dev, logits)
            out.append(logits.clone())
        torch.cuda.synchronize()
        m.set_timing(False)
        return out

    graph = run(False)
    eager = run(True)
    assert m.get_error() == 0
    for s in range(steps):
        assert torch.equal(graph[s], eager[s]), s
        g = graph[s].cpu().numpy()
        assert np.isfinite(g).all(), s
        assert rel_l2(g, refs[s]) <= 2e-2, (s, rel_l2(g, refs[s]))
    m.close()
