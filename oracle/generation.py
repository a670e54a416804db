"""Batched-generation semantics on top of the oracle's general forward pass.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): only tests, the smoke check and the
benchmark's CPU-baseline leg may use it.

Everything here is a choice of (position, cache slot, mask) for each token, handed to
``Model.forward_masked``; no model arithmetic lives in this file. Sources, all on the page
"A modern architecture: Qwen3" (inference.shantanugoel.com/17-qwen3):

* section on generation with a batch of prompts (the ``generate`` function): prompts are padded on
  the left so every row's last token sits in the same column; padding receives no attention;
  positions are counted from each row's first real token (the cumulative count of real tokens,
  minus one, clamped at zero); every token may attend to itself, so a pure-padding row never has
  an empty softmax; decode steps extend the real-token mask by one column and advance each row's
  position by one; a finished row keeps emitting the stop id; generation stops when every row is
  finished, and each row is cut at its first stop id.
* section 8 (prefix caching, ``make_prefix``): the keys and values of a shared start are computed
  once, for one row, at positions 0..P-1 with a causal mask, and every row of the batch starts
  from a copy; the shared slots count as real tokens.
* section 7 (sliding-window attention): token i sees token j iff i - W < j <= i; a rolling buffer of
  W slots writes token i into slot i mod W and attends to every slot it holds, with no mask.

The cache follows the pages' ``Cache``: a token's K/V slot is its column in the concatenated
sequence (prefix columns first), not its position.
"""
from __future__ import annotations

import numpy as np


def left_pad(prompts, pad_id: int, start: int = 0, width: int | None = None):
    """Left-pad a batch of token lists after a shared start of ``start`` slots, to ``width`` columns
    (default: the longest prompt).

    Returns ids [B, width] int32, real [B, start + width] bool, positions [B, width] int32 and
    mask [B, width, start + width] bool (query column t is cache column start + t)."""
    B = len(prompts)
    width = width or max(len(p) for p in prompts)
    if width < max(len(p) for p in prompts):
        raise ValueError("width shorter than a prompt")
    ids = np.full((B, width), pad_id, dtype=np.int32)
    real = np.zeros((B, start + width), dtype=bool)
    real[:, :start] = True
    for b, p in enumerate(prompts):
        if len(p) == 0:
            raise ValueError("empty prompt")
        ids[b, width - len(p):] = p
        real[b, start + width - len(p):] = True
    positions = np.maximum(np.cumsum(real, axis=1) - 1, 0)[:, start:].astype(np.int32)
    qcol = start + np.arange(width)[:, None]
    kcol = np.arange(start + width)[None, :]
    causal = kcol <= qcol
    itself = kcol == qcol
    mask = (causal[None, :, :] & real[:, None, :]) | itself[None, :, :]
    return ids, real, positions, mask


def make_prefix(model, prefix_ids):
    """K/V of a shared start, one row, positions 0..P-1, causal mask (section 8)."""
    P = len(prefix_ids)
    kc, vc = model.new_cache(1, P)
    ids = np.asarray(prefix_ids, dtype=np.int32)[None, :]
    t = np.arange(P)
    model.forward_masked(kc, vc, ids, t[None, :], t[None, :], (t[None, :] <= t[:, None])[None])
    return {"k": kc, "v": vc, "length": P}


def greedy(logits, done, stop_id: int):
    """Next ids: argmax (first index on ties); finished rows emit stop_id. Returns (next, done)."""
    nxt = np.argmax(logits, axis=1).astype(np.int32)
    if done is not None:
        nxt = np.where(done, np.int32(stop_id), nxt)
        done = done | (nxt == stop_id)
    else:
        done = nxt == stop_id
    return nxt, done


def generate(model, prompts, max_new: int, stop_id: int, prefix=None, capacity: int | None = None,
             forced=None, keep=False, pad_id: int | None = None):
    """Greedy generation for a batch of prompts of different lengths.

    Returns (rows, steps): rows = each row's generated ids cut at its first stop id; steps = list of
    dicts per forward call with the logits [B, V], the ids fed, the positions and the cache column.
    ``forced`` (list of [B] arrays) replaces the fed ids of decode step k (teacher forcing) without
    changing the recorded greedy choices. With ``keep`` the final cache is returned in steps[-1].
    Padding uses the stop id, as the pages do, unless ``pad_id`` is given (needed when stop_id < 0
    means "no stop id")."""
    B = len(prompts)
    start = 0 if prefix is None else prefix["length"]
    ids, real, positions, mask = left_pad(prompts, stop_id if pad_id is None else pad_id, start)
    width = ids.shape[1]
    cap = capacity or (start + width + max_new)
    kc, vc = model.new_cache(B, cap)
    if prefix is not None:
        kc[:, :, :, :start] = prefix["k"][:, :1, :, :start]
        vc[:, :, :, :start] = prefix["v"][:, :1, :, :start]
    full = np.zeros((B, width, cap), dtype=bool)
    full[:, :, :start + width] = mask
    slots = (start + np.arange(width, dtype=np.int32))[None, :]
    logits = model.forward_masked(kc, vc, ids, positions, slots, full)
    steps = [dict(logits=logits, ids=ids, positions=positions, column=start)]
    nxt, done = greedy(logits, None, stop_id)
    written = [nxt]
    pos = positions[:, -1].astype(np.int32)
    col = start + width
    real = list(real.T)  # columns
    for k in range(max_new - 1):
        if bool(done.all()):
            break
        pos = pos + 1
        real.append(np.ones(B, dtype=bool))
        m = np.zeros((B, 1, cap), dtype=bool)
        m[:, 0, :col + 1] = np.stack(real, axis=1)
        feed = nxt if forced is None else np.asarray(forced[k], dtype=np.int32)
        logits = model.forward_masked(kc, vc, feed[:, None], pos[:, None], np.int32(col), m)
        steps.append(dict(logits=logits, ids=feed[:, None], positions=pos[:, None], column=col))
        nxt, done = greedy(logits, done, stop_id)
        written.append(nxt)
        col += 1
    if keep:
        steps[-1]["cache"] = (kc, vc)
    table = np.stack(written, axis=1)
    rows = []
    for r in table.tolist():
        rows.append(r[:r.index(stop_id)] if stop_id in r else r)
    return rows, steps


def band_mask(T: int, W: int, start: int = 0):
    """[T, start + T] bool: query start + i sees key j iff start + i - W < j <= start + i (section 7)."""
    q = start + np.arange(T)[:, None]
    k = np.arange(start + T)[None, :]
    return (k <= q) & (q - k < W)


def banded(model, ids, W: int, capacity: int | None = None):
    """One sequence, full causal cache, banded mask; logits of every row."""
    ids = np.asarray(ids, dtype=np.int32).reshape(1, -1)
    T = ids.shape[1]
    cap = capacity or T
    kc, vc = model.new_cache(1, cap)
    m = np.zeros((1, T, cap), dtype=bool)
    m[0, :, :T] = band_mask(T, W)
    t = np.arange(T, dtype=np.int32)[None, :]
    return model.forward_masked(kc, vc, ids, t, t, m, all_rows=True)


def rolling_stepwise(model, ids, W: int):
    """One sequence token by token through a rolling buffer of W slots (slot = i mod W), each step
    attending to every slot written so far; logits of every step [T, V]."""
    ids = np.asarray(ids, dtype=np.int32).reshape(-1)
    kc, vc = model.new_cache(1, W)
    out = []
    for i, tok in enumerate(ids):
        m = np.zeros((1, 1, W), dtype=bool)
        m[0, 0, :min(i + 1, W)] = True
        out.append(model.forward_masked(kc, vc, np.array([[tok]], np.int32), np.int32(i), np.int32(i % W), m))
    return np.concatenate(out, axis=0)
