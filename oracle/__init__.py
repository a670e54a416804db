"""Qwen3 decoder oracle: ctypes wrapper over the plain C++ implementation in qwen3_oracle.cpp.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import this package. It shares no code with the CUDA library and never calls
it. All arrays are numpy; bf16 values travel as their uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qwen3_oracle.cpp")
_LIB = os.path.join(_HERE, "_build", "libqwen3_oracle.so")

_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u8p = ctypes.POINTER(ctypes.c_uint8)


class OracleConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "intermediate", "vocab",
        "tie_embeddings")] + [("rope_theta", ctypes.c_double), ("rms_eps", ctypes.c_double)]


_LAYER_FIELDS = ("in_norm", "q_proj", "k_proj", "v_proj", "o_proj", "q_norm", "k_norm",
                 "post_norm", "gate_proj", "up_proj", "down_proj")


class OracleWeights(ctypes.Structure):
    _fields_ = [("embed", _u16p), ("lm_head", _u16p), ("final_norm", _u16p)] + [
        (n, ctypes.POINTER(_u16p)) for n in _LAYER_FIELDS]


def build(force: bool = False, defines=(), out: str | None = None) -> str:
    """Compile the oracle into a shared library (portable C++17, no ISA flags, no FMA contraction).

    ``defines`` switch on planted mistakes (ORACLE_PLANT_*) for the tests that prove each pin
    catches one; the default build has none.
    """
    out = out or _LIB
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if force or defines or not os.path.exists(out) or os.path.getmtime(out) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "qwen3_oracle.h"))):
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off"]
        cmd += [f"-D{d}" for d in defines]
        subprocess.check_call(cmd + ["-o", out, _SRC])
    return out


_lib = None


def use_library(path: str | None):
    """Point this module at another build of the oracle (a planted variant), or back (None)."""
    global _lib
    _lib = None if path is None else _declare(ctypes.CDLL(path))


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _declare(L: ctypes.CDLL) -> ctypes.CDLL:
    L.oracle_bf16_from_f32.restype = ctypes.c_uint16
    L.oracle_bf16_from_f32.argtypes = [ctypes.c_float]
    L.oracle_bf16_from_f64.restype = ctypes.c_uint16
    L.oracle_bf16_from_f64.argtypes = [ctypes.c_double]
    L.oracle_f32_from_bf16.restype = ctypes.c_float
    L.oracle_f32_from_bf16.argtypes = [ctypes.c_uint16]
    L.oracle_rmsnorm_core_f32.argtypes = [_f32p, ctypes.c_int, ctypes.c_double, _f32p]
    L.oracle_rmsnorm.argtypes = [_u16p, _u16p, ctypes.c_int64, ctypes.c_int, ctypes.c_double, _u16p]
    L.oracle_linear.argtypes = [_u16p, _u16p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _u16p]
    L.oracle_linear_f32out.argtypes = [_u16p, _u16p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _f32p]
    L.oracle_residual_add.argtypes = [_u16p, _u16p, ctypes.c_int64, _u16p]
    L.oracle_silu.restype = ctypes.c_double
    L.oracle_silu.argtypes = [ctypes.c_double]
    L.oracle_swiglu.argtypes = [_u16p, _u16p, ctypes.c_int64, _u16p]
    L.oracle_rope_inv_freq.argtypes = [ctypes.c_double, ctypes.c_int, _f32p]
    L.oracle_rope_cos_sin.argtypes = [ctypes.c_int64, _f32p, ctypes.c_int, _u16p, _u16p]
    L.oracle_rope_apply.argtypes = [_u16p, ctypes.c_int, _u16p, _u16p]
    L.oracle_rope_rotate_f64.argtypes = [_f64p, ctypes.c_int, ctypes.c_double, _f64p, _f64p]
    L.oracle_attention_row_f64.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int64, ctypes.c_int,
                                           ctypes.c_int64, ctypes.c_double, _f64p]
    L.oracle_attention_gqa_row_f64.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int64, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int64, _f64p]
    L.oracle_param_count.argtypes = [ctypes.POINTER(OracleConfig), _i64p]
    L.oracle_layer_qkv.argtypes = [ctypes.POINTER(OracleConfig), ctypes.POINTER(OracleWeights),
                                   ctypes.c_int, _u16p, _i32p, ctypes.c_int64, _u16p, _u16p, _u16p]
    L.oracle_layer_out.argtypes = [ctypes.POINTER(OracleConfig), ctypes.POINTER(OracleWeights),
                                   ctypes.c_int, _u16p, _u16p, _i32p, ctypes.c_int64, _u16p,
                                   _u16p, _i32p, ctypes.c_int64, _u16p]
    L.oracle_head.argtypes = [ctypes.POINTER(OracleConfig), ctypes.POINTER(OracleWeights),
                              _u16p, ctypes.c_int64, _f32p]
    L.oracle_forward.restype = ctypes.c_int
    L.oracle_forward.argtypes = [ctypes.POINTER(OracleConfig), ctypes.POINTER(OracleWeights),
                                 _u16p, _u16p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                 _i32p, ctypes.c_int, ctypes.c_int, _f32p, ctypes.c_int,
                                 _u16p, _u16p]
    L.oracle_attention_masked_gqa_row_f64.restype = ctypes.c_int
    L.oracle_attention_masked_gqa_row_f64.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int64, _u8p, ctypes.c_int,
                                                      ctypes.c_int, ctypes.c_int, _f64p]
    L.oracle_layer_out_masked.restype = ctypes.c_int
    L.oracle_layer_out_masked.argtypes = [ctypes.POINTER(OracleConfig), ctypes.POINTER(OracleWeights), ctypes.c_int,
                                          _u16p, _u16p, ctypes.c_int64, _u16p, _u16p, _i32p, ctypes.c_int64, _u8p,
                                          _u16p]
    L.oracle_forward_masked.restype = ctypes.c_int
    L.oracle_forward_masked.argtypes = [ctypes.POINTER(OracleConfig), ctypes.POINTER(OracleWeights),
                                        _u16p, _u16p, ctypes.c_int, ctypes.c_int64, _i32p, ctypes.c_int,
                                        _i32p, _i32p, _u8p, ctypes.c_int, _f32p, ctypes.c_int, _u16p, _u16p]
    return L


def _p(a: np.ndarray, t):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(t)


def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


# ---------------------------------------------------------------- scalar / elementwise helpers

def bf16_from_f32(x: np.ndarray) -> np.ndarray:
    f = lib().oracle_bf16_from_f32
    x = np.asarray(x, dtype=np.float32)
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def bf16_from_f64(x: np.ndarray) -> np.ndarray:
    f = lib().oracle_bf16_from_f64
    x = np.asarray(x, dtype=np.float64)
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def f32_from_bf16(h: np.ndarray) -> np.ndarray:
    """Bit reinterpretation, the exact widening of a bf16 pattern (no oracle arithmetic)."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def rmsnorm_core_f32(x, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty_like(x)
    lib().oracle_rmsnorm_core_f32(_p(x, _f32p), x.shape[-1], eps, _p(y, _f32p))
    return y


def rmsnorm(x, gamma, eps: float) -> np.ndarray:
    x, gamma = _u16(x), _u16(gamma)
    n = x.shape[-1]
    y = np.empty_like(x)
    lib().oracle_rmsnorm(_p(x, _u16p), _p(gamma, _u16p), x.size // n, n, eps, _p(y, _u16p))
    return y


def linear(a, w, f32_out: bool = False) -> np.ndarray:
    a, w = _u16(a), _u16(w)
    K = a.shape[-1]
    M = a.size // K
    N = w.shape[0]
    assert w.shape[1] == K
    if f32_out:
        y = np.empty(a.shape[:-1] + (N,), dtype=np.float32)
        lib().oracle_linear_f32out(_p(a, _u16p), _p(w, _u16p), M, N, K, _p(y, _f32p))
    else:
        y = np.empty(a.shape[:-1] + (N,), dtype=np.uint16)
        lib().oracle_linear(_p(a, _u16p), _p(w, _u16p), M, N, K, _p(y, _u16p))
    return y


def residual_add(x, y) -> np.ndarray:
    x, y = _u16(x), _u16(y)
    out = np.empty_like(x)
    lib().oracle_residual_add(_p(x, _u16p), _p(y, _u16p), x.size, _p(out, _u16p))
    return out


def silu(z: float) -> float:
    return lib().oracle_silu(float(z))


def swiglu(g, u) -> np.ndarray:
    g, u = _u16(g), _u16(u)
    a = np.empty_like(g)
    lib().oracle_swiglu(_p(g, _u16p), _p(u, _u16p), g.size, _p(a, _u16p))
    return a


def rope_inv_freq(theta: float, dim: int) -> np.ndarray:
    inv = np.empty(dim // 2, dtype=np.float32)
    lib().oracle_rope_inv_freq(theta, dim, _p(inv, _f32p))
    return inv


def rope_cos_sin(pos: int, inv: np.ndarray):
    inv = np.ascontiguousarray(inv, dtype=np.float32)
    c = np.empty(inv.size, dtype=np.uint16)
    s = np.empty(inv.size, dtype=np.uint16)
    lib().oracle_rope_cos_sin(int(pos), _p(inv, _f32p), inv.size, _p(c, _u16p), _p(s, _u16p))
    return c, s


def rope_apply(x, cos_t, sin_t) -> np.ndarray:
    """Rotate each row of x (last dim = head_dim) with one position's bf16 tables."""
    y = _u16(x).copy()
    cos_t, sin_t = _u16(cos_t), _u16(sin_t)
    dim = y.shape[-1]
    flat = y.reshape(-1, dim)
    for r in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[r])
        lib().oracle_rope_apply(_p(row, _u16p), dim, _p(cos_t, _u16p), _p(sin_t, _u16p))
        flat[r] = row
    return flat.reshape(y.shape)


def rope_rotate_f64(x, pos: float, omega) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    omega = np.ascontiguousarray(omega, dtype=np.float64)
    y = np.empty_like(x)
    lib().oracle_rope_rotate_f64(_p(x, _f64p), x.size, float(pos), _p(omega, _f64p), _p(y, _f64p))
    return y


def attention_row_f64(q, k, v, scale: float) -> np.ndarray:
    q, k, v = _u16(q), _u16(k), _u16(v)
    out = np.empty(q.size, dtype=np.float64)
    lib().oracle_attention_row_f64(_p(q, _u16p), _p(k, _u16p), _p(v, _u16p), k.shape[0], q.size,
                                   k.shape[1], scale, _p(out, _f64p))
    return out


def attention_gqa_row_f64(q, kc, vc, n: int) -> np.ndarray:
    """q [Hq, dh] of one row against keys 0..n-1 of kc/vc [Hkv, cap, dh]; returns [Hq, dh] fp64."""
    q, kc, vc = _u16(q), _u16(kc), _u16(vc)
    hq, dim = q.shape
    hkv, cap, _ = kc.shape
    out = np.empty((hq, dim), dtype=np.float64)
    lib().oracle_attention_gqa_row_f64(_p(q, _u16p), _p(kc, _u16p), _p(vc, _u16p), n, hq, hkv, dim,
                                       cap, _p(out, _f64p))
    return out


def attention_masked_gqa_row_f64(q, kc, vc, mask) -> np.ndarray:
    """q [Hq, dh] against the slots of kc/vc [Hkv, cap, dh] that mask [cap] admits; [Hq, dh] fp64."""
    q, kc, vc = _u16(q), _u16(kc), _u16(vc)
    mask = np.ascontiguousarray(mask, dtype=np.uint8)
    hq, dim = q.shape
    hkv, cap, _ = kc.shape
    out = np.empty((hq, dim), dtype=np.float64)
    rc = lib().oracle_attention_masked_gqa_row_f64(_p(q, _u16p), _p(kc, _u16p), _p(vc, _u16p), cap,
                                                   _p(mask, _u8p), hq, hkv, dim, _p(out, _f64p))
    if rc != 0:
        raise ValueError("the mask admits no key")
    return out


# ---------------------------------------------------------------- model

def make_config(cfg: dict) -> OracleConfig:
    return OracleConfig(cfg["n_layers"], cfg["hidden"], cfg["n_q_heads"], cfg["n_kv_heads"],
                        cfg["head_dim"], cfg["intermediate"], cfg["vocab"],
                        int(cfg["tie_embeddings"]), float(cfg["rope_theta"]), float(cfg["rms_eps"]))


def param_count(cfg: dict) -> dict:
    parts = np.zeros(6, dtype=np.int64)
    c = make_config(cfg)
    lib().oracle_param_count(ctypes.byref(c), _p(parts, _i64p))
    names = ("embedding", "attention", "qk_norm", "feed_forward", "other_norms", "lm_head")
    return dict(zip(names, (int(v) for v in parts)))


class Model:
    """Holds host (numpy uint16) weights for the oracle.

    ``weights`` maps names to arrays: embed, lm_head (absent when tied), final_norm, and per-layer
    lists in_norm, q_proj, k_proj, v_proj, o_proj, q_norm, k_norm, post_norm, gate_proj, up_proj,
    down_proj. Layers that are None are not available (sampled checks load only some layers).
    """

    def __init__(self, cfg: dict, weights: dict):
        self.cfg = cfg
        self.c = make_config(cfg)
        self.w = {k: (_u16(v) if isinstance(v, np.ndarray) else v) for k, v in weights.items()}
        L = cfg["n_layers"]
        null = ctypes.cast(None, _u16p)
        arrays = {}
        for name in _LAYER_FIELDS:
            arr = (_u16p * L)()
            lst = self.w[name]
            for i in range(L):
                if lst[i] is not None:
                    lst[i] = _u16(lst[i])
                    arr[i] = _p(lst[i], _u16p)
                else:
                    arr[i] = null
            arrays[name] = arr
        self._arrays = arrays
        lm = self.w.get("lm_head")
        self.ow = OracleWeights(
            _p(self.w["embed"], _u16p) if self.w.get("embed") is not None else null,
            _p(lm, _u16p) if lm is not None else null,
            _p(self.w["final_norm"], _u16p),
            *[ctypes.cast(arrays[n], ctypes.POINTER(_u16p)) for n in _LAYER_FIELDS])

    def new_cache(self, batch: int, capacity: int):
        c = self.cfg
        shape = (c["n_layers"], batch, c["n_kv_heads"], capacity, c["head_dim"])
        return np.zeros(shape, dtype=np.uint16), np.zeros(shape, dtype=np.uint16)

    def forward(self, kc, vc, ids, len0: int, all_rows: bool = False, tap_layer: int = -1):
        """ids [B, T] int32. Returns logits ([B*T, V] or [B, V]) and, when tapping, (in, out)."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        B, T = ids.shape
        cap = kc.shape[3]
        V, d = self.cfg["vocab"], self.cfg["hidden"]
        logits = np.empty(((B * T) if all_rows else B, V), dtype=np.float32)
        tin = np.empty((B * T, d), dtype=np.uint16) if tap_layer >= 0 else None
        tout = np.empty((B * T, d), dtype=np.uint16) if tap_layer >= 0 else None
        null = ctypes.cast(None, _u16p)
        rc = lib().oracle_forward(ctypes.byref(self.c), ctypes.byref(self.ow), _p(kc, _u16p),
                                  _p(vc, _u16p), B, cap, len0, _p(ids, _i32p), T, int(all_rows),
                                  _p(logits, _f32p), tap_layer,
                                  _p(tin, _u16p) if tin is not None else null,
                                  _p(tout, _u16p) if tout is not None else null)
        if rc != 0:
            raise ValueError({-1: "token id out of range", -2: "cache capacity exceeded"}.get(rc, rc))
        return (logits, tin, tout) if tap_layer >= 0 else logits

    def forward_masked(self, kc, vc, ids, pos, slot, mask, all_rows: bool = False, tap_layer: int = -1):
        """General forward: ids, pos, slot [B, T] int32; mask [B, T, cap] bool over cache slots.

        Token (b, t) is rotated at pos[b, t], writes its K/V into slot[b, t] of sequence b and attends to
        the slots mask[b, t] admits (after this call's writes). Returns logits like ``forward``."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        B, T = ids.shape
        cap = kc.shape[3]
        pos = np.ascontiguousarray(np.broadcast_to(pos, (B, T)), dtype=np.int32)
        slot = np.ascontiguousarray(np.broadcast_to(slot, (B, T)), dtype=np.int32)
        mask = np.ascontiguousarray(np.broadcast_to(mask, (B, T, cap)), dtype=np.uint8)
        V, d = self.cfg["vocab"], self.cfg["hidden"]
        logits = np.empty(((B * T) if all_rows else B, V), dtype=np.float32)
        tin = np.empty((B * T, d), dtype=np.uint16) if tap_layer >= 0 else None
        tout = np.empty((B * T, d), dtype=np.uint16) if tap_layer >= 0 else None
        null = ctypes.cast(None, _u16p)
        rc = lib().oracle_forward_masked(ctypes.byref(self.c), ctypes.byref(self.ow), _p(kc, _u16p),
                                         _p(vc, _u16p), B, cap, _p(ids, _i32p), T, _p(pos, _i32p),
                                         _p(slot, _i32p), _p(mask, _u8p), int(all_rows), _p(logits, _f32p),
                                         tap_layer, _p(tin, _u16p) if tin is not None else null,
                                         _p(tout, _u16p) if tout is not None else null)
        if rc != 0:
            raise ValueError({-1: "token id out of range", -2: "cache slot out of range",
                              -3: "a row's mask admits no key"}.get(rc, rc))
        return (logits, tin, tout) if tap_layer >= 0 else logits

    def layer_qkv(self, layer: int, xin, pos):
        c = self.cfg
        xin = _u16(xin)
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        n = xin.shape[0]
        q = np.empty((n, c["n_q_heads"], c["head_dim"]), dtype=np.uint16)
        k = np.empty((n, c["n_kv_heads"], c["head_dim"]), dtype=np.uint16)
        v = np.empty_like(k)
        lib().oracle_layer_qkv(ctypes.byref(self.c), ctypes.byref(self.ow), layer, _p(xin, _u16p),
                               _p(pos, _i32p), n, _p(q, _u16p), _p(k, _u16p), _p(v, _u16p))
        return q, k, v

    def layer_out(self, layer: int, xin, q, pos, kc, vc, kvset):
        """kc/vc: [nsets, Hkv, cap, dh] for this layer."""
        xin, q, kc, vc = _u16(xin), _u16(q), _u16(kc), _u16(vc)
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        kvset = np.ascontiguousarray(kvset, dtype=np.int32)
        n = xin.shape[0]
        out = np.empty_like(xin)
        lib().oracle_layer_out(ctypes.byref(self.c), ctypes.byref(self.ow), layer, _p(xin, _u16p),
                               _p(q, _u16p), _p(pos, _i32p), n, _p(kc, _u16p), _p(vc, _u16p),
                               _p(kvset, _i32p), kc.shape[2], _p(out, _u16p))
        return out

    def layer_out_masked(self, layer: int, xin, q, kc, vc, kvset, mask):
        """Steps a5-a9 with explicit masks: kc/vc [nsets, Hkv, cap, dh]; mask [n, cap] bool over slots."""
        xin, q, kc, vc = _u16(xin), _u16(q), _u16(kc), _u16(vc)
        kvset = np.ascontiguousarray(kvset, dtype=np.int32)
        mask = np.ascontiguousarray(mask, dtype=np.uint8)
        n = xin.shape[0]
        out = np.empty_like(xin)
        rc = lib().oracle_layer_out_masked(ctypes.byref(self.c), ctypes.byref(self.ow), layer, _p(xin, _u16p),
                                           _p(q, _u16p), n, _p(kc, _u16p), _p(vc, _u16p), _p(kvset, _i32p),
                                           kc.shape[2], _p(mask, _u8p), _p(out, _u16p))
        if rc != 0:
            raise ValueError("a row's mask admits no key")
        return out

    def head(self, x):
        x = _u16(x)
        n = x.shape[0]
        logits = np.empty((n, self.cfg["vocab"]), dtype=np.float32)
        lib().oracle_head(ctypes.byref(self.c), ctypes.byref(self.ow), _p(x, _u16p), n, _p(logits, _f32p))
        return logits
