"""ctypes binding of the C ABI in include/qwen3.h. Argument marshalling only: every step of the
forward pass runs in the CUDA library; torch tensors only provide device memory and streams.

The library must have been built (``__graft_entry__.build()``); loading fails loudly otherwise.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from .build import LIB

_vp = ctypes.c_void_p
_i32p = ctypes.POINTER(ctypes.c_int)

EPI_BF16, EPI_SWIGLU, EPI_RESIDUAL, EPI_F32 = 0, 1, 2, 3
ALL_ROWS = 1


class Qwen3Error(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what} (code {code})")
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "intermediate", "vocab",
        "tie_embeddings", "max_positions")] + [("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float),
                                               ("sliding_window", ctypes.c_int32), ("rolling_cache", ctypes.c_int32)]

    @classmethod
    def from_dict(cls, c: dict) -> "Config":
        return cls(c["n_layers"], c["hidden"], c["n_q_heads"], c["n_kv_heads"], c["head_dim"],
                   c["intermediate"], c["vocab"], int(c["tie_embeddings"]), c.get("max_positions", 40960),
                   float(c["rope_theta"]), float(c["rms_eps"]), int(c.get("sliding_window", 0)),
                   int(c.get("rolling_cache", 0)))


_LAYER = ("in_norm", "q_proj", "k_proj", "v_proj", "o_proj", "q_norm", "k_norm", "post_norm", "gate_proj",
          "up_proj", "down_proj")


class Weights(ctypes.Structure):
    _fields_ = [("embed", _vp), ("lm_head", _vp), ("final_norm", _vp)] + [(n, ctypes.POINTER(_vp)) for n in _LAYER]


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB):
        raise RuntimeError(f"CUDA library not built ({LIB}); run __graft_entry__.build() first")
    L = ctypes.CDLL(LIB)
    i, sz, cp = ctypes.c_int, ctypes.c_size_t, ctypes.c_char_p
    L.qwen3_strerror.restype = cp
    L.qwen3_strerror.argtypes = [i]
    L.qwen3_validate_config.argtypes = [ctypes.POINTER(Config)]
    L.qwen3_init.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights), i, i, i, _vp, ctypes.POINTER(_vp)]
    L.qwen3_prefill.argtypes = [_vp, _vp, i, i, _vp, i, _vp]
    L.qwen3_decode_step.argtypes = [_vp, _vp, i, _vp, _vp]
    L.qwen3_prefill_host.argtypes = [_vp, _vp, i, i, _vp, i, _vp]
    L.qwen3_length.argtypes = [_vp, _i32p, _i32p]
    L.qwen3_set_length.argtypes = [_vp, i, i, _vp]
    L.qwen3_kv_view.argtypes = [_vp, i, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(ctypes.c_int64)]
    L.qwen3_set_tap.argtypes = [_vp, i, _vp, _vp]
    L.qwen3_get_error.argtypes = [_vp, _vp]
    L.qwen3_set_timing.argtypes = [_vp, i]
    L.qwen3_kernel_times.argtypes = [_vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64), _i32p]
    L.qwen3_kernel_class_name.restype = cp
    L.qwen3_kernel_class_name.argtypes = [i]
    L.qwen3_launch_count.argtypes = [_vp, i, i, i, i]
    L.qwen3_free.restype = None
    L.qwen3_free.argtypes = [_vp]
    L.qwen3_op_embed.argtypes = [_vp, i, i, _vp, i, _vp, _vp, _vp]
    L.qwen3_op_rmsnorm.argtypes = [_vp, _vp, i, i, i, i, ctypes.c_float, _vp, _vp]
    L.qwen3_op_gemm.argtypes = [_vp, _vp, i, i, i, i, _vp, i, _vp, i, _vp, _vp]
    L.qwen3_op_pack_gate_up.argtypes = [_vp, _vp, i, i, _vp, _vp]
    L.qwen3_gemm_norm_supported.argtypes = [i, i]
    L.qwen3_gemm_norm_part_floats.restype = sz
    L.qwen3_gemm_norm_part_floats.argtypes = [i]
    L.qwen3_op_gemm_residual_norm.argtypes = [_vp, _vp, i, i, i, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp]
    L.qwen3_gemm_skinny_splits.argtypes = [i, i]
    L.qwen3_op_gemm_skinny.argtypes = [_vp, _vp, i, i, i, i, _vp, _vp, _vp, _vp]
    L.qwen3_op_rope_table.argtypes = [ctypes.c_float, i, i, _vp, _vp]
    L.qwen3_op_qknorm_rope_append.argtypes = [_vp, i, i, i, i, i, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp,
                                              _vp, i, _vp]
    L.qwen3_op_attention_prefill.argtypes = [_vp, _vp, _vp, i, i, i, i, i, i, _vp, _vp, i, i, i, i, i, _vp, _vp,
                                             _vp, _vp]
    L.qwen3_attention_prefill_workspace.restype = sz
    L.qwen3_attention_prefill_workspace.argtypes = [i, i, i, i, i, i]
    L.qwen3_attention_decode_workspace.restype = sz
    L.qwen3_attention_decode_workspace.argtypes = [i, i, i, i, i, i]
    L.qwen3_op_attention_decode.argtypes = [_vp, _vp, _vp, i, i, i, i, i, _vp, _vp, i, i, _vp, _vp, _vp, _vp]
    L.qwen3_op_attention_decode_noalloc.argtypes = [_vp, _vp, _vp, i, i, i, i, i, _vp, _vp, _vp, _vp]
    L.qwen3_op_greedy.argtypes = [_vp, ctypes.c_int64, i, i, i, _vp, _vp, _vp, _vp]
    L.qwen3_greedy_workspace.restype = sz
    L.qwen3_greedy_workspace.argtypes = [i]
    L.qwen3_prefill_padded.argtypes = [_vp, _vp, _i32p, i, i, _vp, i, _vp]
    L.qwen3_share_prefix.argtypes = [_vp, i, _vp]
    L.qwen3_generate.argtypes = [_vp, _vp, _i32p, i, i, i, i, _vp, _i32p, _vp]
    _lib = L
    return L


def strerror(code: int) -> str:
    return lib().qwen3_strerror(code).decode()


def check(rc: int):
    if rc != 0:
        raise Qwen3Error(rc, strerror(rc))


def _p(t) -> _vp:
    if t is None:
        return _vp(None)
    if isinstance(t, np.ndarray):
        return _vp(t.ctypes.data)
    return _vp(t.data_ptr())


def _stream(stream=None) -> _vp:
    s = torch.cuda.current_stream() if stream is None else stream
    return _vp(s.cuda_stream)


class _DeviceArray:
    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"data": (ptr, False), "shape": tuple(shape), "typestr": typestr,
                                         "version": 3, "strides": None}


def device_view(ptr: int, shape, dtype) -> torch.Tensor:
    """A torch tensor that aliases device memory owned by the library (no copy)."""
    if dtype == torch.bfloat16:
        return torch.as_tensor(_DeviceArray(ptr, shape, "<i2"), device="cuda").view(torch.bfloat16)
    typestr = {torch.float32: "<f4", torch.int32: "<i4"}[dtype]
    return torch.as_tensor(_DeviceArray(ptr, shape, typestr), device="cuda")


def validate_config(cfg: dict) -> int:
    c = Config.from_dict(cfg)
    return lib().qwen3_validate_config(ctypes.byref(c))


class Model:
    """A Qwen3 decoder context: KV cache, scratch and packed weights owned by the library.

    ``weights`` holds bf16 CUDA tensors in nn.Linear layout (synth.make_weights format); they are
    borrowed and kept alive by this object.
    """

    def __init__(self, cfg: dict, weights: dict, max_batch: int, capacity: int, max_tokens: int = 0,
                 stream=None):
        self.cfg = cfg
        self._w = weights
        L = cfg["n_layers"]
        self._arrays = {}
        for name in _LAYER:
            arr = (_vp * L)(*[t.data_ptr() for t in weights[name]])
            self._arrays[name] = arr
        lm = weights.get("lm_head")
        self._ws = Weights(_p(weights["embed"]), _p(lm), _p(weights["final_norm"]),
                           *[ctypes.cast(self._arrays[n], ctypes.POINTER(_vp)) for n in _LAYER])
        self._cfg = Config.from_dict(cfg)
        self.ctx = _vp()
        check(lib().qwen3_init(ctypes.byref(self._cfg), ctypes.byref(self._ws), max_batch, capacity, max_tokens,
                               _stream(stream), ctypes.byref(self.ctx)))
        self.max_batch, self.capacity = max_batch, capacity

    def close(self):
        if self.ctx:
            lib().qwen3_free(self.ctx)
            self.ctx = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, ids: torch.Tensor, logits: torch.Tensor, all_rows: bool = False, stream=None):
        B, T = ids.shape
        check(lib().qwen3_prefill(self.ctx, _p(ids), B, T, _p(logits), ALL_ROWS if all_rows else 0,
                                  _stream(stream)))

    def prefill_padded(self, ids: torch.Tensor, real, logits: torch.Tensor, all_rows: bool = False, stream=None):
        """ids [B, T] left-padded; real[b] = number of real tokens at the end of row b."""
        B, T = ids.shape
        r = (ctypes.c_int32 * B)(*[int(x) for x in real])
        check(lib().qwen3_prefill_padded(self.ctx, _p(ids), r, B, T, _p(logits), ALL_ROWS if all_rows else 0,
                                         _stream(stream)))

    def share_prefix(self, batch: int, stream=None):
        check(lib().qwen3_share_prefix(self.ctx, batch, _stream(stream)))

    def generate(self, ids: torch.Tensor, real, max_new: int, stop_id: int, out: torch.Tensor, stream=None) -> int:
        """Greedy generation; out [B, max_new] int32 receives the tokens. Returns the columns written."""
        B, T = ids.shape
        r = (ctypes.c_int32 * B)(*[int(x) for x in real]) if real is not None else None
        steps = ctypes.c_int32()
        check(lib().qwen3_generate(self.ctx, _p(ids), r, B, T, max_new, stop_id, _p(out), ctypes.byref(steps),
                                   _stream(stream)))
        return steps.value

    def decode_step(self, ids: torch.Tensor, logits: torch.Tensor, stream=None):
        check(lib().qwen3_decode_step(self.ctx, _p(ids), ids.shape[0], _p(logits), _stream(stream)))

    def prefill_host(self, ids: np.ndarray, logits: np.ndarray, all_rows: bool = False, stream=None):
        B, T = ids.shape
        check(lib().qwen3_prefill_host(self.ctx, _p(ids), B, T, _p(logits), ALL_ROWS if all_rows else 0,
                                       _stream(stream)))

    def length(self):
        n, b = ctypes.c_int(), ctypes.c_int()
        check(lib().qwen3_length(self.ctx, ctypes.byref(n), ctypes.byref(b)))
        return n.value, b.value

    def set_length(self, length: int, batch: int, stream=None):
        check(lib().qwen3_set_length(self.ctx, length, batch, _stream(stream)))

    def kv_view(self, layer: int):
        k, v = _vp(), _vp()
        dims = (ctypes.c_int64 * 4)()
        check(lib().qwen3_kv_view(self.ctx, layer, ctypes.byref(k), ctypes.byref(v), dims))
        shape = tuple(dims)
        return device_view(k.value, shape, torch.bfloat16), device_view(v.value, shape, torch.bfloat16)

    def set_tap(self, layer: int, t_in: torch.Tensor | None = None, t_out: torch.Tensor | None = None):
        check(lib().qwen3_set_tap(self.ctx, layer, _p(t_in), _p(t_out)))

    def get_error(self, stream=None) -> int:
        return lib().qwen3_get_error(self.ctx, _stream(stream))

    def set_timing(self, enable: bool):
        check(lib().qwen3_set_timing(self.ctx, int(enable)))

    def kernel_times(self) -> dict:
        n = ctypes.c_int(32)
        ms = (ctypes.c_double * 32)()
        cnt = (ctypes.c_int64 * 32)()
        check(lib().qwen3_kernel_times(self.ctx, ms, cnt, ctypes.byref(n)))
        return {lib().qwen3_kernel_class_name(i).decode(): (ms[i], cnt[i]) for i in range(n.value)}

    def launch_count(self, B: int, T: int, decode: bool = False, all_rows: bool = False) -> int:
        return lib().qwen3_launch_count(self.ctx, B, T, ALL_ROWS if all_rows else 0, int(decode))


# ------------------------------------------------------------------------------ single operations

def op_embed(E, ids, out, err, stream=None):
    V, d = E.shape
    check(lib().qwen3_op_embed(_p(E), V, d, _p(ids), ids.numel(), _p(out), _p(err), _stream(stream)))


def op_rmsnorm(x, gamma, eps, out, rows=None, in_stride=1, in_offset=0, stream=None):
    n = gamma.numel()
    rows = out.numel() // n if rows is None else rows
    check(lib().qwen3_op_rmsnorm(_p(x), _p(gamma), rows, n, in_stride, in_offset, eps, _p(out), _stream(stream)))


def op_gemm(A, B, epi, C, R=None, err=None, stream=None):
    M, K = A.shape
    N = B.shape[0]
    check(lib().qwen3_op_gemm(_p(A), _p(B), M, N, K, epi, _p(C), C.shape[1], _p(R),
                              R.shape[1] if R is not None else 0, _p(err), _stream(stream)))


def gemm_norm_supported(M, N) -> bool:
    return bool(lib().qwen3_gemm_norm_supported(M, N))


def gemm_norm_part_floats(M) -> int:
    return lib().qwen3_gemm_norm_part_floats(M)


def op_gemm_residual_norm(A, B, X, gamma, eps, Y, part, err=None, stream=None):
    """X [M, N] += A B^T in place (bf16 rounding as QWEN3_EPI_RESIDUAL), Y = RMSNorm(X; gamma)."""
    M, K = A.shape
    N = B.shape[0]
    check(lib().qwen3_op_gemm_residual_norm(_p(A), _p(B), M, N, K, _p(X), _p(gamma), eps, _p(Y), _p(part), _p(err),
                                            _stream(stream)))


def gemm_skinny_splits(N, K) -> int:
    return lib().qwen3_gemm_skinny_splits(N, K)


def op_gemm_skinny(A, B, splits, slices=None, out=None, err=None, stream=None):
    M, K = A.shape
    N = B.shape[0]
    check(lib().qwen3_op_gemm_skinny(_p(A), _p(B), M, N, K, splits, _p(slices), _p(out), _p(err), _stream(stream)))


def op_pack_gate_up(gate, up, out, stream=None):
    F, d = gate.shape
    check(lib().qwen3_op_pack_gate_up(_p(gate), _p(up), F, d, _p(out), _stream(stream)))


def op_rope_table(theta, dh, n_pos, out, stream=None):
    check(lib().qwen3_op_rope_table(theta, dh, n_pos, _p(out), _stream(stream)))


def op_qknorm_rope_append(qkv, B, T, Hq, Hkv, dh, q_gamma, k_gamma, table, len0, eps, q_out, k_cache, v_cache,
                          stream=None):
    cap = k_cache.shape[2]
    check(lib().qwen3_op_qknorm_rope_append(_p(qkv), B, T, Hq, Hkv, dh, _p(q_gamma), _p(k_gamma), _p(table),
                                            _p(len0), eps, _p(q_out), _p(k_cache), _p(v_cache), cap,
                                            _stream(stream)))


def attention_prefill_workspace(B, T, Hq, Hkv, dh, kv_chunks) -> int:
    return lib().qwen3_attention_prefill_workspace(B, T, Hq, Hkv, dh, kv_chunks)


def op_attention_prefill(q, k_cache, v_cache, len0, out, err=None, kv_split=0, kv_chunks=1, work=None,
                         seq_meta=None, window=0, ring=0, heads_per_cta=0, stream=None):
    B, Hq, T, dh = q.shape
    Hkv, cap = k_cache.shape[1], k_cache.shape[2]
    check(lib().qwen3_op_attention_prefill(_p(q), _p(k_cache), _p(v_cache), B, T, Hq, Hkv, dh, cap, _p(len0),
                                           _p(seq_meta), window, ring, heads_per_cta, kv_split, kv_chunks, _p(work),
                                           _p(out), _p(err), _stream(stream)))


def attention_decode_workspace(B, Hq, dh, cap, window=0, ring=0) -> int:
    return lib().qwen3_attention_decode_workspace(B, Hq, dh, cap, window, ring)


def op_attention_decode(q, k_cache, v_cache, len0, work, out, seq_meta=None, window=0, ring=0, err=None,
                        stream=None):
    B, Hq, dh = q.shape
    Hkv, cap = k_cache.shape[1], k_cache.shape[2]
    check(lib().qwen3_op_attention_decode(_p(q), _p(k_cache), _p(v_cache), B, Hq, Hkv, dh, cap, _p(len0),
                                          _p(seq_meta), window, ring, _p(work), _p(out), _p(err), _stream(stream)))


_greedy_work = {}


def greedy_workspace(B) -> int:
    return lib().qwen3_greedy_workspace(B)


def op_greedy(logits, next_ids, stop_id=-1, done=None, work="auto", stream=None):
    """work: "auto" (a zeroed scratch buffer kept per device and size, reused across calls on one stream),
    None (one CTA per row), or a caller tensor of greedy_workspace(B) bytes, zero before its first use."""
    B, V = logits.shape
    if isinstance(work, str):
        key = (logits.device, greedy_workspace(B))
        if key not in _greedy_work:
            _greedy_work[key] = torch.zeros(max(1, key[1] // 4), dtype=torch.int32, device=logits.device)
        work = _greedy_work[key]
    check(lib().qwen3_op_greedy(_p(logits), logits.stride(0), B, V, stop_id, _p(done), _p(next_ids), _p(work),
                                _stream(stream)))
