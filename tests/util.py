"""Shared helpers for the tests: error metrics and host/device conversions (no model arithmetic)."""
import numpy as np
import torch

from qwen3_decoder_transformer_gb300 import synth

bits = synth.to_numpy_bits


def widen(u16: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 values (exact)."""
    return (np.ascontiguousarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rel_l2(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def max_rel_rows(got, ref, width: int) -> float:
    """Largest relative L2 error over consecutive groups of `width` values (e.g. one (row, head) output
    vector of head_dim values each), so that a single wrong row or head cannot hide in an aggregate."""
    g = np.asarray(got, dtype=np.float64).reshape(-1, width)
    r = np.asarray(ref, dtype=np.float64).reshape(-1, width)
    den = np.linalg.norm(r, axis=1)
    num = np.linalg.norm(g - r, axis=1)
    return float(np.max(num / np.where(den > 0, den, 1.0)))


def dev(u16: np.ndarray) -> torch.Tensor:
    """Host bf16 bit patterns -> CUDA bf16 tensor."""
    return synth.from_numpy_bits(u16, "cuda")


def rand_bf16(rng: np.random.Generator, shape, scale=1.0) -> np.ndarray:
    return bits(torch.from_numpy(rng.standard_normal(shape) * scale).to(torch.bfloat16))


def top1_agreement(got: np.ndarray, ref: np.ndarray):
    """Fraction of rows with equal argmax (first index on ties), over all rows and over rows whose
    reference top-1/top-2 margin exceeds 4x the largest absolute logit error seen."""
    g, r = got.argmax(-1), ref.argmax(-1)
    part = np.partition(ref, -2, axis=-1)
    margin = part[:, -1] - part[:, -2]
    err = np.abs(got - ref).max()
    clear = margin > 4 * err
    raw = float((g == r).mean())
    filt = float((g[clear] == r[clear]).mean()) if clear.any() else 1.0
    return raw, filt, int(clear.sum())
