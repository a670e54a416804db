"""The allocation-free decode-attention entry point (qwen3_op_attention_decode_noalloc) must give the
result of the workspace entry point (qwen3_op_attention_decode). It exists for callers that cannot call
cudaMalloc, so its partials live in a fixed array inside the library; this test calls it twice in a row
through the C ABI, with different shapes, and checks both results, and checks that a shape whose
partials do not fit is refused. Collected last so that a run stopping at the first failure has run
every other test."""
import ctypes

import numpy as np
import pytest
import torch

from qwen3_decoder_transformer_gb300 import build as B
from tests.util import bits, dev, rand_bf16, rel_l2, widen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    B.build()
    from qwen3_decoder_transformer_gb300 import binding
    lib = binding.lib()
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.qwen3_op_attention_decode_noalloc.argtypes = [vp, vp, vp, i, i, i, i, i, vp, vp, vp]
    return binding, lib


def _case(seed, Bq, Hq, Hkv, dh, n, cap):
    rng = np.random.default_rng(seed)
    q = dev(rand_bf16(rng, (Bq, Hq, dh)))
    kc = dev(rand_bf16(rng, (Bq, Hkv, cap, dh)))
    vc = dev(rand_bf16(rng, (Bq, Hkv, cap, dh)))
    return q, kc, vc, torch.tensor([n - 1], dtype=torch.int32, device="cuda")


def _noalloc(lib, q, kc, vc, len_t, out):
    Bq, Hq, dh = q.shape
    Hkv, cap = kc.shape[1], kc.shape[2]
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return lib.qwen3_op_attention_decode_noalloc(p(q), p(kc), p(vc), Bq, Hq, Hkv, dh, cap, p(len_t), p(out),
                                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point(L):
    binding, lib = L
    cases = [(1, 4, 16, 8, 128, 4097, 4224), (2, 2, 32, 8, 128, 1000, 1100)]
    for seed, Bq, Hq, Hkv, dh, n, cap in cases:
        q, kc, vc, len_t = _case(seed, Bq, Hq, Hkv, dh, n, cap)
        work = torch.zeros(binding.attention_decode_workspace(Bq, Hq, dh, cap) // 4, dtype=torch.float32,
                           device="cuda")
        ref = torch.empty(Bq, Hq * dh, dtype=torch.bfloat16, device="cuda")
        binding.op_attention_decode(q, kc, vc, len_t, work, ref)
        got = torch.full_like(ref, float("nan"))
        assert _noalloc(lib, q, kc, vc, len_t, got) == 0
        torch.cuda.synchronize()
        g, r = widen(bits(got)), widen(bits(ref))
        assert np.isfinite(g).all()
        assert rel_l2(g, r) <= 1e-2


def test_noalloc_refuses_oversized_workspace(L):
    binding, lib = L
    Bq, Hq, Hkv, dh, cap = 64, 32, 8, 128, 32832
    assert binding.attention_decode_workspace(Bq, Hq, dh, cap) > (16 << 20)
    q = torch.zeros(Bq, Hq, dh, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(1, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(Bq, Hq * dh, dtype=torch.bfloat16, device="cuda")
    len_t = torch.zeros(1, dtype=torch.int32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.qwen3_op_attention_decode_noalloc(p(q), p(kc), p(kc), Bq, Hq, Hkv, dh, cap, p(len_t), p(out),
                                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 5  # QWEN3_E_ARG, nothing launched
