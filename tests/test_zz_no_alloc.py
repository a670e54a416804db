"""The allocation-free decode-attention entry point (qwen3_op_attention_decode_noalloc) against the workspace
entry point (qwen3_op_attention_decode) and the oracle.

Some callers cannot call cudaMalloc: their device memory belongs to another allocator, or an allocation's
implicit device synchronisation is not allowed, or nothing may be allocated after start-up. For them the
split partials live in a fixed array inside the library that every call shares and that keeps whatever the
last call left there. The calls below run in a row on that one array: the first leaves NaN partials (a NaN
value in the cache) and records of chunks past a later call's length; the later calls, with other lengths
and other shapes, must not read any of it. Each result must equal the workspace entry point's bit for bit
(both run the same kernels; the workspace there starts as NaN) and match the oracle's brute-force GQA row
within the attention tolerance. Collected last so that a run stopping at the first failure has run every
other test; it passes alone in a fresh process too.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from qwen3_decoder_transformer_gb300 import build as B
from tests.util import bits, dev, max_rel_rows, rand_bf16, rel_l2, widen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    B.build()
    from qwen3_decoder_transformer_gb300 import binding
    return binding, binding.lib()


def _noalloc(lib, q, kc, vc, len_t, out, err):
    Bq, Hq, dh = q.shape
    Hkv, cap = kc.shape[1], kc.shape[2]
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return lib.qwen3_op_attention_decode_noalloc(p(q), p(kc), p(vc), Bq, Hq, Hkv, dh, cap, p(len_t), p(out), p(err),
                                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _run_both(binding, lib, q, kc, vc, n):
    """(allocation-free result, workspace result) as bf16 bit patterns."""
    Bq, Hq, dh = q.shape
    cap = kc.shape[2]
    len_t = torch.tensor([n - 1], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    work = torch.full((binding.attention_decode_workspace(Bq, Hq, dh, cap) // 4,), float("nan"), dtype=torch.float32,
                      device="cuda")
    ref = torch.empty(Bq, Hq * dh, dtype=torch.bfloat16, device="cuda")
    binding.op_attention_decode(q, kc, vc, len_t, work, ref, err=err)
    got = torch.empty_like(ref)
    assert _noalloc(lib, q, kc, vc, len_t, got, err) == 0
    torch.cuda.synchronize()
    assert err.item() == 0
    return bits(got), bits(ref)


def test_noalloc_matches_workspace_entry_point_and_oracle(L):
    binding, lib = L
    rng = np.random.default_rng(7)
    # call 1: 2 x 16 heads, dh 128, 4097 keys in 512-slot chunks; one V value in chunk 5 of sequence 0,
    # kv head 0 is NaN, so the partials of that chunk (query heads 0 and 1) are NaN
    Bq, Hq, Hkv, dh, cap = 2, 16, 8, 128, 4224
    q = rand_bf16(rng, (Bq, Hq, dh))
    kc = rand_bf16(rng, (Bq, Hkv, cap, dh))
    vc = rand_bf16(rng, (Bq, Hkv, cap, dh))
    vc[0, 0, 3000, 5] = 0x7FC0
    qd, kd, vd = dev(q), dev(kc), dev(vc)
    got, ref = _run_both(binding, lib, qd, kd, vd, 4097)
    assert np.array_equal(got, ref)
    g = widen(got).reshape(Bq, Hq, dh)
    assert np.isnan(g[0, :2]).any() and np.isfinite(g[0, 2:]).all() and np.isfinite(g[1]).all()

    # call 2: the same caches with 1000 keys (chunks 0 and 1): chunk 5's NaN partials stay in the array
    # from call 1 and must not be read
    got, ref = _run_both(binding, lib, qd, kd, vd, 1000)
    assert np.array_equal(got, ref)
    o = np.stack([O.attention_gqa_row_f64(q[b], kc[b], vc[b], 1000).ravel() for b in range(Bq)])
    gw = widen(got)
    assert np.isfinite(gw).all()
    assert rel_l2(gw, o) <= 1e-2 and max_rel_rows(gw, o, dh) <= 3e-2

    # call 3: another shape (4 x 32 heads, dh 64, 1024-slot chunks of a 17,000-slot cache): its records sit
    # at other offsets of the array, over what calls 1 and 2 left there, and 16 of its 17 chunks hold no key
    Bq, Hq, Hkv, dh, cap, n = 4, 32, 8, 64, 17000, 1500
    q = rand_bf16(rng, (Bq, Hq, dh))
    kc = rand_bf16(rng, (Bq, Hkv, cap, dh))
    vc = rand_bf16(rng, (Bq, Hkv, cap, dh))
    kc[:, :, n:] = 0x7FC0
    vc[:, :, n:] = 0x7FC0
    got, ref = _run_both(binding, lib, dev(q), dev(kc), dev(vc), n)
    assert np.array_equal(got, ref)
    o = np.stack([O.attention_gqa_row_f64(q[b], kc[b], vc[b], n).ravel() for b in range(Bq)])
    gw = widen(got)
    assert np.isfinite(gw).all()
    assert rel_l2(gw, o) <= 1e-2 and max_rel_rows(gw, o, dh) <= 3e-2


def test_noalloc_refuses_oversized_workspace(L):
    binding, lib = L
    Bq, Hq, Hkv, dh, cap = 64, 32, 8, 128, 32832
    assert binding.attention_decode_workspace(Bq, Hq, dh, cap) > (16 << 20)
    q = torch.zeros(Bq, Hq, dh, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(1, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(Bq, Hq * dh, dtype=torch.bfloat16, device="cuda")
    len_t = torch.zeros(1, dtype=torch.int32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.qwen3_op_attention_decode_noalloc(p(q), p(kc), p(kc), Bq, Hq, Hkv, dh, cap, p(len_t), p(out), None,
                                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 5  # QWEN3_E_ARG, nothing launched
