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
