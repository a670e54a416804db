"""Per-kernel parity: each CUDA kernel, called through the C ABI's single-operation entry points, against
the oracle on the same seeded inputs. Shapes span several tiles plus ragged tails.

Tolerances (relative L2 unless stated): gather and cache indexing bit-exact; RMSNorm, RoPE table and
q/k-norm+RoPE 1e-3; GEMM epilogues 1e-3 (bf16 outputs) and 1e-5 (fp32 logits); attention 1e-2 over the
whole output (P is rounded to bf16 on the tensor cores, the oracle keeps it exact) and 3e-2 for every
single (row, head) output vector, so that one wrong row or head cannot hide in the aggregate.
"""
import numpy as np
import pytest
import torch

import oracle as O
from qwen3_decoder_transformer_gb300 import build as B
from tests.util import bits, dev, max_rel_rows, rand_bf16, rel_l2, widen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bd():
    B.build()
    from qwen3_decoder_transformer_gb300 import binding
    binding.lib()
    return binding


def _err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ------------------------------------------------------------------------------------ embedding

def test_embed_bitexact(bd):
    rng = np.random.default_rng(0)
    V, d = 1000, 256
    E = rand_bf16(rng, (V, d), 0.02)
    ids = rng.integers(0, V, 301).astype(np.int32)
    out = torch.empty(301, d, dtype=torch.bfloat16, device="cuda")
    err = _err()
    bd.op_embed(dev(E), torch.from_numpy(ids).cuda(), out, err)
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), E[ids])
    assert err.item() == 0


def test_embed_bad_id_zeroes_row_and_flags(bd):
    rng = np.random.default_rng(1)
    E = rand_bf16(rng, (64, 128), 0.02)
    ids = np.array([3, 64, -1, 5], dtype=np.int32)
    out = torch.full((4, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    err = _err()
    bd.op_embed(dev(E), torch.from_numpy(ids).cuda(), out, err)
    torch.cuda.synchronize()
    got = bits(out)
    assert np.array_equal(got[0], E[3]) and np.array_equal(got[3], E[5])
    assert not got[1].any() and not got[2].any()
    assert err.item() & 1


# -------------------------------------------------------------------------------------- RMSNorm

@pytest.mark.parametrize("rows,n", [(1, 256), (7, 1024), (300, 4096), (33, 64), (5, 8192), (1000, 1024)])
def test_rmsnorm(bd, rows, n):
    rng = np.random.default_rng(rows * 7 + n)
    x = rand_bf16(rng, (rows, n), 3.0)
    g = bits(torch.from_numpy(1 + 0.2 * (rng.random(n) - 0.5)).to(torch.bfloat16))
    y = torch.empty(rows, n, dtype=torch.bfloat16, device="cuda")
    bd.op_rmsnorm(dev(x), dev(g), 1e-6, y)
    torch.cuda.synchronize()
    ref = O.rmsnorm(x, g, 1e-6)
    got = bits(y)
    assert rel_l2(widen(got), widen(ref)) <= 1e-3
    assert (got == ref).mean() > 0.99


def test_rmsnorm_last_row_selection(bd):
    rng = np.random.default_rng(5)
    Bq, T, n = 3, 17, 1024
    x = rand_bf16(rng, (Bq * T, n))
    g = bits(torch.ones(n, dtype=torch.bfloat16))
    y = torch.empty(Bq, n, dtype=torch.bfloat16, device="cuda")
    bd.op_rmsnorm(dev(x), dev(g), 1e-6, y, rows=Bq, in_stride=T, in_offset=T - 1)
    torch.cuda.synchronize()
    ref = O.rmsnorm(x[T - 1::T], g, 1e-6)
    assert rel_l2(widen(bits(y)), widen(ref)) <= 1e-3


# ------------------------------------------------------------------------------------ RoPE table

@pytest.mark.parametrize("dh", [64, 128])
def test_rope_table(bd, dh):
    n_pos = 32832
    tab = torch.empty(n_pos, dh, dtype=torch.bfloat16, device="cuda")
    bd.op_rope_table(1e6, dh, n_pos, tab)
    torch.cuda.synchronize()
    got = bits(tab)
    inv = O.rope_inv_freq(1e6, dh)
    positions = list(range(0, 70)) + list(range(4090, 4230)) + list(range(32700, n_pos)) + [12345, 23456]
    ref = np.stack([np.concatenate(O.rope_cos_sin(p, inv)) for p in positions])
    assert rel_l2(widen(got[positions]), widen(ref)) <= 1e-3
    assert (got[positions] == ref).mean() > 0.999


# ------------------------------------------------------------------------- q/k norm + RoPE + append

@pytest.mark.parametrize("Bq,T,Hq,Hkv,dh,len0", [(1, 64, 8, 4, 64, 0), (2, 37, 16, 8, 128, 5),
                                                  (3, 1, 32, 8, 128, 4095)])
def test_qknorm_rope_append(bd, Bq, T, Hq, Hkv, dh, len0):
    rng = np.random.default_rng(Bq * 100 + T)
    cap = len0 + T + 3
    H = Hq + 2 * Hkv
    qkv = rand_bf16(rng, (Bq * T, H * dh), 2.0)
    qg = bits(torch.from_numpy(1 + 0.2 * (rng.random(dh) - 0.5)).to(torch.bfloat16))
    kg = bits(torch.from_numpy(1 + 0.2 * (rng.random(dh) - 0.5)).to(torch.bfloat16))
    table = torch.empty(cap, dh, dtype=torch.bfloat16, device="cuda")
    bd.op_rope_table(1e6, dh, cap, table)
    len_t = torch.tensor([len0], dtype=torch.int32, device="cuda")
    q_out = torch.empty(Bq, Hq, T, dh, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(Bq, Hkv, cap, dh, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    bd.op_qknorm_rope_append(dev(qkv), Bq, T, Hq, Hkv, dh, dev(qg), dev(kg), table, len_t, 1e-6, q_out, kc, vc)
    torch.cuda.synchronize()
    inv = O.rope_inv_freq(1e6, dh)
    x = qkv.reshape(Bq, T, H, dh)
    q_ref = np.empty((Bq, Hq, T, dh), np.uint16)
    k_ref = np.zeros((Bq, Hkv, cap, dh), np.uint16)
    v_ref = np.zeros((Bq, Hkv, cap, dh), np.uint16)
    for t in range(T):
        c, s = O.rope_cos_sin(len0 + t, inv)
        qn = O.rmsnorm(np.ascontiguousarray(x[:, t, :Hq]), qg, 1e-6)
        kn = O.rmsnorm(np.ascontiguousarray(x[:, t, Hq:Hq + Hkv]), kg, 1e-6)
        q_ref[:, :, t] = O.rope_apply(qn, c, s)
        k_ref[:, :, len0 + t] = O.rope_apply(kn, c, s)
        v_ref[:, :, len0 + t] = x[:, t, Hq + Hkv:]
    got_k, got_v = bits(kc), bits(vc)
    assert np.array_equal(got_v, v_ref)  # V copied bit-exactly into the right slots, nothing else written
    mask = np.zeros(cap, bool)
    mask[len0:len0 + T] = True
    assert not got_k[:, :, ~mask].any()  # untouched slots stay zero
    assert rel_l2(widen(got_k), widen(k_ref)) <= 1e-3
    assert rel_l2(widen(bits(q_out)), widen(q_ref)) <= 1e-3
    assert (bits(q_out) == q_ref).mean() > 0.99


# ------------------------------------------------------------------------------------------ GEMM

GEMM_SHAPES = [(1, 256, 64), (64, 512, 256), (200, 1024, 1024), (300, 768, 512), (129, 2048, 192)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_gemm_bf16(bd, M, N, K):
    rng = np.random.default_rng(M + N + K)
    a = rand_bf16(rng, (M, K))
    w = rand_bf16(rng, (N, K), 0.05)
    c = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    err = _err()
    bd.op_gemm(dev(a), dev(w), bd.EPI_BF16, c, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref = O.linear(a, w)
    got = bits(c)
    assert rel_l2(widen(got), widen(ref)) <= 1e-3
    assert (got == ref).mean() > 0.98


@pytest.mark.parametrize("M,N,K", [(5, 1000, 256), (130, 1000, 1024), (64, 151936 // 8, 256)])
def test_gemm_f32_ragged_n(bd, M, N, K):
    rng = np.random.default_rng(N + M)
    a = rand_bf16(rng, (M, K))
    w = rand_bf16(rng, (N, K), 0.05)
    c = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    bd.op_gemm(dev(a), dev(w), bd.EPI_F32, c)
    torch.cuda.synchronize()
    ref = O.linear(a, w, f32_out=True)
    assert rel_l2(c.cpu().numpy(), ref) <= 1e-5


@pytest.mark.parametrize("M,F,K", [(1, 128, 64), (200, 768, 256), (257, 1536, 512)])
def test_gemm_swiglu(bd, M, F, K):
    rng = np.random.default_rng(M * F)
    a = rand_bf16(rng, (M, K))
    wg = rand_bf16(rng, (F, K), 0.08)
    wu = rand_bf16(rng, (F, K), 0.08)
    packed = torch.empty(2 * F, K, dtype=torch.bfloat16, device="cuda")
    bd.op_pack_gate_up(dev(wg), dev(wu), packed)
    c = torch.empty(M, F, dtype=torch.bfloat16, device="cuda")
    bd.op_gemm(dev(a), packed, bd.EPI_SWIGLU, c)
    torch.cuda.synchronize()
    ref = O.swiglu(O.linear(a, wg), O.linear(a, wu))
    assert rel_l2(widen(bits(c)), widen(ref)) <= 1e-3


@pytest.mark.parametrize("M,N,K", [(3, 256, 512), (200, 1024, 2048), (129, 512, 3072)])
def test_gemm_residual_in_place(bd, M, N, K):
    rng = np.random.default_rng(M + 3 * N)
    a = rand_bf16(rng, (M, K))
    w = rand_bf16(rng, (N, K), 0.02)
    x = rand_bf16(rng, (M, N))
    xd = dev(x)
    bd.op_gemm(dev(a), dev(w), bd.EPI_RESIDUAL, xd, R=xd)
    torch.cuda.synchronize()
    ref = O.residual_add(x, O.linear(a, w))
    assert rel_l2(widen(bits(xd)), widen(ref)) <= 1e-3


@pytest.mark.parametrize("M,N,K", [(3, 256, 512), (200, 1024, 2048), (2048, 1024, 1024), (129, 512, 3072),
                                   (5000, 1024, 512)])
def test_gemm_residual_norm(bd, M, N, K):
    """Residual GEMM fused with the next RMSNorm: X against the oracle's residual add, Y against the
    oracle's RMSNorm of the kernel's own X (each stage pinned on its own). 5000 x 1024 takes 256-wide
    tiles (4 per row block), the others 128-wide ones (N / 128 per row block)."""
    assert bd.gemm_norm_supported(M, N)
    rng = np.random.default_rng(M + 5 * N)
    a = rand_bf16(rng, (M, K))
    w = rand_bf16(rng, (N, K), 0.02)
    x = rand_bf16(rng, (M, N))
    g = bits(torch.from_numpy(1 + 0.2 * (rng.random(N) - 0.5)).to(torch.bfloat16))
    xd, y = dev(x), torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    part = torch.zeros(bd.gemm_norm_part_floats(M), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.op_gemm_residual_norm(dev(a), dev(w), xd, dev(g), 1e-6, y, part, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    got_x = bits(xd)
    assert rel_l2(widen(got_x), widen(O.residual_add(x, O.linear(a, w)))) <= 1e-3
    got_y, ref_y = bits(y), O.rmsnorm(got_x, g, 1e-6)
    assert rel_l2(widen(got_y), widen(ref_y)) <= 1e-3
    assert (got_y == ref_y).mean() > 0.99
    # the meeting counters are left zero for the next call
    rows_blocks = (M + 127) // 128
    assert not part.view(torch.int32)[rows_blocks * 16 * 128:].any()


def test_gemm_residual_norm_unsupported_shape(bd):
    """More than 8 column tiles per row block are not supported: refused, nothing launched."""
    assert not bd.gemm_norm_supported(64, 4096)
    a, w = torch.zeros(64, 256, dtype=torch.bfloat16, device="cuda"), torch.zeros(4096, 256, dtype=torch.bfloat16,
                                                                                    device="cuda")
    x, y = torch.zeros(64, 4096, dtype=torch.bfloat16, device="cuda"), torch.zeros(64, 4096, dtype=torch.bfloat16,
                                                                                   device="cuda")
    g, part = torch.ones(4096, dtype=torch.bfloat16, device="cuda"), torch.zeros(4096, dtype=torch.float32,
                                                                                 device="cuda")
    with pytest.raises(bd.Qwen3Error):
        bd.op_gemm_residual_norm(a, w, x, g, 1e-6, y, part)


@pytest.mark.parametrize("M,N,K", [(1, 256, 64), (16, 4096, 4096), (64, 1024, 2048), (5, 1000, 1024), (33, 3072, 512)])
def test_gemm_skinny(bd, M, N, K):
    """Decode GEMM: split-K slices (summed on the test side) and the unsplit direct store."""
    rng = np.random.default_rng(M * 7 + N)
    a = rand_bf16(rng, (M, K))
    w = rand_bf16(rng, (N, K), 0.05)
    ref = O.linear(a, w, f32_out=True)
    splits = bd.gemm_skinny_splits(N, K)
    err = _err()
    if splits > 1:
        sl = torch.full((splits, M, N), float("nan"), dtype=torch.float32, device="cuda")
        bd.op_gemm_skinny(dev(a), dev(w), splits, slices=sl, err=err)
        torch.cuda.synchronize()
        assert rel_l2(sl.sum(0).double().cpu().numpy(), ref) <= 1e-5
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    bd.op_gemm_skinny(dev(a), dev(w), 1, out=out, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert rel_l2(out.cpu().numpy(), ref) <= 1e-5


# ------------------------------------------------------------------------------------- attention

def _attn_ref(q, kc, vc, len0, T):
    """q [B,Hq,T,dh] bits; caches [B,Hkv,cap,dh] bits -> [B*T, Hq*dh] fp64 via the oracle."""
    Bq, Hq, _, dh = q.shape
    out = np.empty((Bq, T, Hq * dh))
    for b in range(Bq):
        for t in range(T):
            out[b, t] = O.attention_gqa_row_f64(np.ascontiguousarray(q[b, :, t]), kc[b], vc[b], len0 + t + 1).ravel()
    return out.reshape(Bq * T, Hq * dh)


@pytest.mark.parametrize("Bq,T,Hq,Hkv,dh,len0", [(1, 64, 8, 4, 64, 0), (2, 130, 8, 2, 64, 0),
                                                  (1, 200, 16, 8, 128, 0), (2, 77, 16, 8, 128, 70),
                                                  (1, 1, 4, 4, 128, 300), (1, 700, 8, 2, 128, 0),
                                                  (1, 384, 4, 1, 64, 129), (3, 257, 8, 8, 128, 511)])
def test_attention_prefill(bd, Bq, T, Hq, Hkv, dh, len0):
    _attention_prefill_case(bd, Bq, T, Hq, Hkv, dh, len0, 0, 1)


@pytest.mark.parametrize("Bq,T,Hq,Hkv,dh,len0", [(1, 64, 8, 4, 64, 0), (2, 130, 8, 2, 64, 0), (1, 700, 8, 2, 128, 0),
                                                  (2, 77, 16, 8, 128, 70), (3, 257, 8, 8, 128, 511)])
def test_attention_prefill_one_head_per_cta(bd, Bq, T, Hq, Hkv, dh, len0):
    """The one-head-per-CTA variant (score regions alternate between tiles)."""
    _attention_prefill_case(bd, Bq, T, Hq, Hkv, dh, len0, 0, 1, heads=1)
    if Hkv < Hq:
        _attention_prefill_case(bd, Bq, T, Hq, Hkv, dh, len0, 1, 3, heads=1)


@pytest.mark.parametrize("Bq,T,Hq,Hkv,dh,len0", [(1, 64, 8, 4, 64, 0), (2, 130, 8, 2, 64, 0), (1, 700, 8, 2, 128, 0),
                                                  (2, 77, 16, 8, 128, 70), (3, 257, 8, 2, 128, 511),
                                                  (1, 1100, 4, 2, 128, 1000)])
def test_attention_prefill_two_heads_per_cta(bd, Bq, T, Hq, Hkv, dh, len0):
    """The two-heads-per-CTA kernel without a KV split (the long-prompt kernel; the automatic choice takes it
    only at 16 or more waves of CTAs, so the heads are forced here)."""
    _attention_prefill_case(bd, Bq, T, Hq, Hkv, dh, len0, 0, 1, heads=2)


@pytest.mark.parametrize("Bq,T,Hq,Hkv,dh,len0,split,chunks", [(1, 700, 8, 2, 128, 0, 1, 4), (1, 1024, 16, 8, 128, 0, 2, 4),
                                                               (2, 257, 8, 8, 128, 511, 1, 3), (1, 384, 4, 1, 64, 129, 1, 2),
                                                               (1, 300, 8, 4, 64, 70, 1, 8)])
def test_attention_prefill_split_kv(bd, Bq, T, Hq, Hkv, dh, len0, split, chunks):
    _attention_prefill_case(bd, Bq, T, Hq, Hkv, dh, len0, split, chunks)


def _attention_prefill_case(bd, Bq, T, Hq, Hkv, dh, len0, split, chunks, heads=0):
    rng = np.random.default_rng(T * 31 + len0)
    cap = len0 + T + 5
    q = rand_bf16(rng, (Bq, Hq, T, dh))
    kc = rand_bf16(rng, (Bq, Hkv, cap, dh))
    vc = rand_bf16(rng, (Bq, Hkv, cap, dh))
    kc[:, :, len0 + T:] = 0x7FC0  # NaN past the written slots: must never be read
    vc[:, :, len0 + T:] = 0x7FC0
    out = torch.empty(Bq * T, Hq * dh, dtype=torch.bfloat16, device="cuda")
    len_t = torch.tensor([len0], dtype=torch.int32, device="cuda")
    err = _err()
    work = None
    if split:
        work = torch.zeros(max(1, bd.attention_prefill_workspace(Bq, T, Hq, Hkv, dh, chunks) // 4),
                           dtype=torch.float32, device="cuda")
    for _ in range(2 if split else 1):  # twice: the merge tickets must be left at zero
        bd.op_attention_prefill(dev(q), dev(kc), dev(vc), len_t, out, err=err, kv_split=split, kv_chunks=chunks,
                                work=work, heads_per_cta=heads)
    torch.cuda.synchronize()
    assert err.item() == 0
    if split:
        assert not work[:64].view(torch.int32).any()
    ref = _attn_ref(q, kc, vc, len0, T)
    got = widen(bits(out))
    assert np.isfinite(got).all()
    assert rel_l2(got, ref) <= 1e-2
    assert max_rel_rows(got, ref, dh) <= 3e-2


@pytest.mark.parametrize("Bq,Hq,Hkv,dh,n,extra", [(1, 8, 4, 64, 1, 40), (3, 16, 8, 128, 300, 40),
                                                   (2, 32, 8, 128, 1000, 40), (4, 16, 8, 128, 4097, 40),
                                                   (1, 8, 8, 128, 257, 40), (2, 16, 8, 128, 300, 3800),
                                                   (1, 8, 2, 64, 70, 20000)])
def test_attention_decode(bd, Bq, Hq, Hkv, dh, n, extra):
    """Decode attention against the oracle's brute-force GQA row. The workspace starts as NaN and cache
    slots past the length hold NaN: neither may reach the output. `extra` slots of capacity past the
    length give chunks with no key at all (a roomy cache), which the merge must not read."""
    rng = np.random.default_rng(n + Hq)
    cap = n + extra
    q = rand_bf16(rng, (Bq, Hq, dh))
    kc = rand_bf16(rng, (Bq, Hkv, cap, dh))
    vc = rand_bf16(rng, (Bq, Hkv, cap, dh))
    kc[:, :, n:] = 0x7FC0
    vc[:, :, n:] = 0x7FC0
    work = torch.full((bd.attention_decode_workspace(Bq, Hq, dh, cap) // 4,), float("nan"), dtype=torch.float32,
                      device="cuda")
    out = torch.empty(Bq, Hq * dh, dtype=torch.bfloat16, device="cuda")
    len_t = torch.tensor([n - 1], dtype=torch.int32, device="cuda")
    err = _err()
    bd.op_attention_decode(dev(q), dev(kc), dev(vc), len_t, work, out, err=err)
    first = out.clone()
    work.fill_(float("inf"))
    bd.op_attention_decode(dev(q), dev(kc), dev(vc), len_t, work, out, err=err)  # same result over any workspace
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(first, out)
    ref = np.stack([O.attention_gqa_row_f64(q[b], kc[b], vc[b], n).ravel() for b in range(Bq)])
    got = widen(bits(out))
    assert np.isfinite(got).all()
    assert rel_l2(got, ref) <= 1e-2
    assert max_rel_rows(got, ref, dh) <= 3e-2


@pytest.mark.parametrize("T,window,dh,len0", [(16384 + 77, 0, 128, 0), (16500, 1000, 128, 0), (16384 + 77, 0, 64, 0),
                                               (16384 + 77, 0, 128, 300), (8192 + 5, 0, 128, 0)])
def test_attention_prefill_long_keys(bd, T, window, dh, len0):
    """Key ranges of 8192 and more take the alternating form of the persistent kernel: two softmax
    warpgroups take alternate key tiles and hand each row's scale from tile to tile; the exponentials start
    with the scale known so far and are recomputed when it moved. With a sliding window, rows of one warp
    reach their first visible key at different tiles; with len0 cached tokens the block's query t sees
    slots 0..len0 + t (a chunk after a prefix). Sampled rows against the oracle's brute-force row, per-row
    bounds included; slots past the block hold NaN."""
    rng = np.random.default_rng(T + window + dh + len0)
    Bq, Hq, Hkv = 1, 4, 2
    n = len0 + T
    cap = n + 3
    q = rand_bf16(rng, (Bq, Hq, T, dh))
    kc = rand_bf16(rng, (Bq, Hkv, cap, dh))
    vc = rand_bf16(rng, (Bq, Hkv, cap, dh))
    kc[:, :, n:] = 0x7FC0
    vc[:, :, n:] = 0x7FC0
    out = torch.empty(Bq * T, Hq * dh, dtype=torch.bfloat16, device="cuda")
    len_t = torch.tensor([len0], dtype=torch.int32, device="cuda")
    err = _err()
    bd.op_attention_prefill(dev(q), dev(kc), dev(vc), len_t, out, err=err, window=window)
    torch.cuda.synchronize()
    assert err.item() == 0
    got = widen(bits(out)).reshape(T, Hq * dh)
    rows = sorted(r for r in {0, 1, 127, 128, 999, 1000, 1001, 5000, 8191, 12345, 16383, T - 2, T - 1} if r < T)
    for t in rows:
        p = len0 + t  # the query's own slot
        lo = max(0, p + 1 - window) if window else 0
        ref = O.attention_gqa_row_f64(np.ascontiguousarray(q[0, :, t]), np.ascontiguousarray(kc[0][:, lo:p + 1]),
                                      np.ascontiguousarray(vc[0][:, lo:p + 1]), p + 1 - lo).ravel()
        assert np.isfinite(got[t]).all(), t
        assert rel_l2(got[t], ref) <= 1e-2, t
        assert max_rel_rows(got[t], ref, dh) <= 3e-2, t
