"""The C ABI library builds, loads without a GPU, exports every function include/qwen3.h declares,
and rejects bad shapes and arguments on the host."""
import ctypes
import os
import re

import pytest

from qwen3_decoder_transformer_gb300 import QWEN3_0P6B, QWEN3_8B, TINY, build as B
from tests.conftest import ROOT


@pytest.fixture(scope="module")
def L():
    B.build()
    from qwen3_decoder_transformer_gb300 import binding
    return binding.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "qwen3.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qwen3_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(L, n), n


def test_validate_config(L):
    from qwen3_decoder_transformer_gb300 import binding
    for cfg in (TINY, QWEN3_0P6B, QWEN3_8B):
        assert binding.validate_config(cfg) == 0
    bad = [dict(TINY, n_kv_heads=3), dict(TINY, head_dim=96), dict(TINY, hidden=100),
           dict(TINY, intermediate=700), dict(TINY, vocab=1001), dict(TINY, n_layers=0),
           dict(TINY, n_q_heads=24, n_kv_heads=2)]
    for cfg in bad:
        assert binding.validate_config(cfg) == 1, cfg
    assert L.qwen3_validate_config(None) == 5


def test_strerror(L):
    from qwen3_decoder_transformer_gb300 import binding
    assert binding.strerror(0) == "ok"
    assert "capacity" in binding.strerror(3)
    assert "context limit" in binding.strerror(2)
    assert binding.strerror(123) == "unknown error"


def test_host_argument_errors(L):
    from qwen3_decoder_transformer_gb300 import binding
    out = ctypes.c_void_p()
    cfg = binding.Config.from_dict(TINY)
    assert L.qwen3_init(ctypes.byref(cfg), None, 1, 16, 0, None, ctypes.byref(out)) == 5
    assert L.qwen3_prefill(None, None, 1, 1, None, 0, None) == 5
    assert L.qwen3_decode_step(None, None, 1, None, None) == 5
    assert L.qwen3_op_gemm(None, None, 1, 1, 8, 0, None, 8, None, 0, None, None) == 5
    assert L.qwen3_op_rmsnorm(None, None, 1, 8, 1, 0, ctypes.c_float(1e-6), None, None) == 5
    assert L.qwen3_kernel_class_name(0) == b"embed"


def test_decode_workspace_chunk_policy(L):
    """Decode attention splits the cache into chunks of 1024 slots (caches of 16,384+ slots), 512
    (shorter caches) or 256 (a rolling ring); a window needs only the chunks it can touch. The
    workspace holds [m, l, o[dh]] fp32 per (sequence, query head, chunk)."""
    from qwen3_decoder_transformer_gb300 import binding

    def ws(B, Hq, dh, cap, window=0, ring=0):
        return binding.attention_decode_workspace(B, Hq, dh, cap, window, ring)

    rec = lambda dh: (dh + 2) * 4
    assert ws(64, 16, 128, 4096 + 16) == 64 * 16 * 9 * rec(128)        # 512-slot chunks
    assert ws(16, 32, 128, 32768 + 16) == 16 * 32 * 33 * rec(128)      # 1024-slot chunks
    assert ws(16, 32, 128, 32768 + 16, window=4096) == 16 * 32 * 5 * rec(128)
    assert ws(16, 32, 128, 4352, window=4096, ring=4352) == 16 * 32 * 17 * rec(128)  # 256-slot chunks
    assert ws(1, 8, 64, 80) == 1 * 8 * 1 * rec(64)
    assert ws(0, 8, 64, 80) == 0


def test_decode_noalloc_refuses_large_workspace(L):
    """A call whose partials would not fit the library's fixed 16 MiB array is refused on the host
    (QWEN3_E_ARG) before anything is launched."""
    from qwen3_decoder_transformer_gb300 import binding
    assert binding.attention_decode_workspace(64, 32, 128, 32832, 0, 0) > (16 << 20)
    dummy = ctypes.c_void_p(16)  # never dereferenced: the size check comes first
    len0 = ctypes.cast(ctypes.c_void_p(16), ctypes.POINTER(ctypes.c_int))
    assert L.qwen3_op_attention_decode_noalloc(dummy, dummy, dummy, 64, 32, 8, 128, 32832, len0, dummy, None, None) == 5
