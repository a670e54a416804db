// Causal grouped-query attention over the KV cache ("A modern architecture: Qwen3", Attention with
// grouped KV heads and Q/K normalization; "Transformer architectures: modern", section 3: query head
// h reads kv head floor(h / g), g = Hq / Hkv; scores scaled by head_dim^-0.5; causal mask).
//
// Prefill: flash attention with an online softmax on the 5th-generation tensor cores (tcgen05,
// accumulators in tensor memory, operands staged by TMA); see the kernel's own comment.
//
// Decode: one query per (sequence, query head) against the whole cache. A CTA owns a chunk (256 to
// 1024 keys) of one (sequence, kv head) and serves all g query heads of that group from one read of
// K and V, streamed by TMA into shared memory; the scores and the weighted sum run as warp-level
// tensor-core contractions with the group's heads as the narrow dimension. Partial (max, sum,
// output) triples go to a workspace; a second kernel merges the chunks by log-sum-exp.
#include <algorithm>
#include <cfloat>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace q3 {
namespace {


// --------------------------------------------------------------------------- prefill (tcgen05)
// One CTA = 128 query rows of NH query heads that share one kv head. Tensor memory holds two
// 128-column score regions and NH 128-column output accumulators. Warps:
//   warp 0          TMA: the NH Q tiles once, then K_j / V_j tiles (128 keys) into 2-stage rings; a K
//                   stage is refilled as soon as its scores are done, a V stage once its PV is done.
//   warp 1          TMEM owner and MMA issuer. S = Q_h K_j^T into a score region (128 fp32 columns);
//                   softmax overwrites its first 64 columns with P as packed bf16; then O_h += P V_j
//                   reads P straight from TMEM (A operand in tensor memory) and V_j as an MN-major
//                   shared-memory operand. The MMA pipe executes in issue order, which makes a later
//                   S overwriting an earlier P safe.
//                   NH = 2: one region per head; order per tile PV_0, S_0(next), PV_1, S_1(next), so
//                   one head's scores are computed while the other head's softmax runs.
//                   NH = 1: the two regions alternate between tiles, and the scores of tile j+1 are
//                   computed while the softmax of tile j runs (S_{j+2} is issued right after PV_j).
//   warps 2..2+4NH  softmax, four warps per head; thread r owns query row r (TMEM lane r). Online
//                   softmax in base 2 with lazy rescaling: O and l are rescaled only when the running
//                   max grows by more than 8 (so P <= 256). At the end each thread normalises its row.
// Causal mask: key k is visible to query t iff k <= len0 + t; tiles wholly above the diagonal are
// not loaded, and only tiles crossing it are masked. V rows past the last valid key are zeroed in
// shared memory before use so stale cache contents cannot reach O through 0 * NaN.
constexpr int TC_BM = 128, TC_BN = 128, TC_STAGES = 2;

template <int DH, int NH>
struct TcLayout {
    static constexpr int NCH = DH / 64;             // 64-element (128-byte) column chunks
    static constexpr int Q_BYTES = TC_BM * DH * 2;  // per head: [NCH][128 rows][128 B]
    static constexpr int KV_BYTES = TC_BN * DH * 2;
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = NH * Q_BYTES;
    static constexpr int V_OFF = K_OFF + TC_STAGES * KV_BYTES;
    static constexpr int BAR_OFF = V_OFF + TC_STAGES * KV_BYTES;
    static constexpr int SMEM = BAR_OFF + 256 + 1024;
    static constexpr int THREADS = 64 + 128 * NH;
};

template <int DH, int NH>
__global__ void __launch_bounds__(TcLayout<DH, NH>::THREADS, 1)
    attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, int T, int Hq, int Hkv,
                           const int* __restrict__ len0p, const int* __restrict__ meta, int window, int ring,
                           __nv_bfloat16* __restrict__ out, int* err, int split, int max_chunks,
                           float* __restrict__ ws, int* __restrict__ tickets) {
    using Ly = TcLayout<DH, NH>;
    constexpr int NCH = Ly::NCH;
    constexpr uint32_t IDESC_S = idesc_bf16(TC_BM, TC_BN);
    constexpr uint32_t IDESC_O = idesc_bf16(TC_BM, DH, true);
    constexpr uint32_t TM_O = 2 * TC_BN;  // O_h at TM_O + h * 128
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Ly::BAR_OFF);
    uint64_t* q_full = bars;
    uint64_t* k_full = bars + 1;    // [2]
    uint64_t* v_full = bars + 3;    // [2]
    uint64_t* k_empty = bars + 5;   // [2]
    uint64_t* v_empty = bars + 7;   // [2]
    uint64_t* s_full = bars + 9;    // [2] per score region
    uint64_t* p_full = bars + 11;   // [2] per score region
    uint64_t* o_done = bars + 13;   // [NH]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 15);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 16);
    volatile int* merge_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_qt = gridDim.x / max_chunks;
    const int qt = n_qt - 1 - (int)(blockIdx.x / max_chunks);  // longest query tiles first
    const int chunk = (int)(blockIdx.x % max_chunks);
    const int h0 = blockIdx.y * NH, b = blockIdx.z;
    const int jkv = h0 / (Hq / Hkv);
    const int q0 = qt * TC_BM;
    const int q_end = min(T, q0 + TC_BM);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 128);
        }
        for (int hh = 0; hh < NH; ++hh) mbar_init(&o_done[hh], 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;
    pdl_wait();  // Q and the cache come from the previous kernel
    pdl_trigger();
    const int len0 = *len0p;
    // sequence layout: padding slots [ps, pe) of this sequence, slots below psh read from sequence 0
    int ps = 0, pe = 0, psh = 0;
    if (meta) {
        ps = meta[0];
        psh = meta[1];
        pe = ps + meta[kSeqMetaHead + b];
    }
    const int n_valid = len0 + q_end;
    const int n_end = (n_valid + TC_BN - 1) / TC_BN;
    // a sliding window starts at the tile holding the first query's oldest visible key
    const int j_lo = window > 0 ? max(0, len0 + q0 - window + 1) / TC_BN : 0;
    // tiles [ja, jb) lie wholly inside this sequence's padding and below every query of the block:
    // no row sees any of their keys, so they are skipped
    const int ja = max(j_lo, (ps + TC_BN - 1) / TC_BN);
    const int jb = max(ja, min(pe / TC_BN, (len0 + q0) / TC_BN));
    const int n_tiles = n_end - j_lo - (jb - ja);
    // absolute KV tile of the i-th live tile (counted from j_lo)
    auto tile_of_live = [&](int i) { return j_lo + i < ja ? j_lo + i : j_lo + i + (jb - ja); };
    // score region of head hh at this CTA's tile i, and how many earlier tiles used it (barrier phase)
    auto s_region = [](int hh, int i) { return NH == 2 ? hh : (i & 1); };
    auto s_use = [](int i) { return NH == 2 ? i : (i >> 1); };
    // KV range of this CTA: the whole causal range, or one chunk of it (split > 0: chunks of at least
    // `split` tiles, at most max_chunks of them, merged by the last CTA of the query tile to finish)
    const int chunk_tiles = split > 0 ? max(split, (n_tiles + max_chunks - 1) / max_chunks) : n_tiles;
    const int n_chunks = (n_tiles + chunk_tiles - 1) / chunk_tiles;
    const int jc = chunk * chunk_tiles;  // first live tile of this chunk
    const int nt = chunk < n_chunks ? min(n_tiles, jc + chunk_tiles) - jc : 0;  // tiles of this CTA

    if (warp == 0) {
        if (lane == 0 && nt > 0) {
            mbar_expect_tx(q_full, NH * Ly::Q_BYTES);
            for (int hh = 0; hh < NH; ++hh)
                for (int c = 0; c < NCH; ++c)
                    tma_load_3d(smem + Ly::Q_OFF + hh * Ly::Q_BYTES + c * TC_BM * 128, &tmQ, q_full, c * 64, q0,
                                b * Hq + h0 + hh);
            for (int i = 0; i < nt; ++i) {
                const int s = i & 1, j = tile_of_live(jc + i);
                const uint32_t free_ph = ((i >> 1) & 1) ^ 1;
                // cache row of the tile (a rolling buffer wraps) and its sequence (a shared prefix
                // lives in sequence 0)
                const int y = ring ? (j * TC_BN) % ring : j * TC_BN;
                const int z = (j * TC_BN < psh ? 0 : b) * Hkv + jkv;
                if (!mbar_wait_suspend(&k_empty[s], free_ph, abort_flag)) { ok = false; break; }
                mbar_expect_tx(&k_full[s], Ly::KV_BYTES);
                for (int c = 0; c < NCH; ++c)
                    tma_load_3d(smem + Ly::K_OFF + s * Ly::KV_BYTES + c * TC_BN * 128, &tmK, &k_full[s], c * 64, y, z);
                if (!mbar_wait_suspend(&v_empty[s], free_ph, abort_flag)) { ok = false; break; }
                mbar_expect_tx(&v_full[s], Ly::KV_BYTES);
                for (int c = 0; c < NCH; ++c)
                    tma_load_3d(smem + Ly::V_OFF + s * Ly::KV_BYTES + c * TC_BN * 128, &tmV, &v_full[s], c * 64, y, z);
            }
        }
    } else if (warp == 1 && nt > 0) {
        // all lanes walk the schedule (so the warp can zero V tails together); lane 0 issues.
        // i counts this CTA's tiles (barrier phases); j = tile_of_live(jc + i) is the absolute KV tile.
        auto issue_s = [&](int hh, int i) -> bool {
            const int s = i & 1;
            if (!__all_sync(0xffffffffu, mbar_wait_suspend(&k_full[s], (i >> 1) & 1, abort_flag))) return false;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t sq = smem_u32(smem + Ly::Q_OFF + hh * Ly::Q_BYTES);
                const uint32_t sk = smem_u32(smem + Ly::K_OFF + s * Ly::KV_BYTES);
                const int r = s_region(hh, i);
#pragma unroll
                for (int kk = 0; kk < DH / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * TC_BM * 128 + (kk & 3) * 32;
                    umma_bf16_ss(tmem + r * TC_BN, sdesc_kmajor_sw128(sq + off), sdesc_kmajor_sw128(sk + off), IDESC_S,
                                 kk > 0);
                }
                umma_commit(&s_full[r]);
                if (hh == NH - 1) umma_commit(&k_empty[s]);  // K_i is no longer needed
            }
            __syncwarp();
            return true;
        };
        ok = __all_sync(0xffffffffu, mbar_wait_suspend(q_full, 0, abort_flag));
        // scores run ahead: tile 0 of both heads (NH = 2), or tiles 0 and 1 (NH = 1)
        for (int hh = 0; ok && hh < NH; ++hh) ok = issue_s(hh, 0);
        if (NH == 1 && ok && nt > 1) ok = issue_s(0, 1);
        for (int i = 0; ok && i < nt; ++i) {
            const int s = i & 1, j = tile_of_live(jc + i);
            if (!__all_sync(0xffffffffu, mbar_wait_suspend(&v_full[s], (i >> 1) & 1, abort_flag))) { ok = false; break; }
            uint8_t* sv = smem + Ly::V_OFF + s * Ly::KV_BYTES;
            const int r0 = n_valid - j * TC_BN;  // first stale key row of this tile
            if (r0 < TC_BN) {
                for (int i = lane; i < (TC_BN - r0) * 8 * NCH; i += 32) {
                    const int c = i / ((TC_BN - r0) * 8), rem = i % ((TC_BN - r0) * 8);
                    reinterpret_cast<uint4*>(sv + c * TC_BN * 128 + (r0 + rem / 8) * 128)[rem % 8] =
                        make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            for (int hh = 0; ok && hh < NH; ++hh) {
                const int r = s_region(hh, i);
                if (!__all_sync(0xffffffffu, mbar_wait_suspend(&p_full[r], s_use(i) & 1, abort_flag))) { ok = false; break; }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t svv = smem_u32(sv);
#pragma unroll
                    for (int kk = 0; kk < TC_BN / 16; ++kk) {
                        const uint64_t bd = sdesc_mnmajor_sw128(svv + kk * 16 * 128, TC_BN * 128);
                        umma_bf16_ts(tmem + TM_O + hh * 128, tmem + r * TC_BN + kk * 8, bd, IDESC_O, (i | kk) != 0);
                    }
                    umma_commit(&o_done[hh]);
                    if (hh == NH - 1) umma_commit(&v_empty[s]);  // V_i is no longer needed
                }
                __syncwarp();
                const int nxt = NH == 2 ? i + 1 : i + 2;  // the next tile whose scores go to region r
                if (nxt < nt) ok = issue_s(hh, nxt);
            }
        }
    } else if (warp >= 2 && nt > 0) {
        // softmax warps: head hh, thread <-> query row
        const int hh = (warp - 2) >> 2;
        const int quarter = warp & 3, row = quarter * 32 + lane;
        const int t = q0 + row, pos = len0 + t;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tm_o = tmem + lane_off + TM_O + hh * 128;
        const float sl2 = kLog2e / sqrtf((float)DH);
        float m_used = -INFINITY, l = 0.f;  // m_used in scaled (log2) units
        int pv_seen = 0;                    // PV completions confirmed so far
        auto confirm_pv = [&](int upto) -> bool {
            while (pv_seen < upto) {
                if (!mbar_wait_suspend(&o_done[hh], pv_seen & 1, abort_flag)) return false;
                ++pv_seen;
            }
            return true;
        };
        for (int i = 0; i < nt; ++i) {
            const int j = tile_of_live(jc + i);
            const int r = s_region(hh, i);
            const uint32_t tm_s = tmem + lane_off + r * TC_BN;
            if (!__all_sync(0xffffffffu, mbar_wait_suspend(&s_full[r], s_use(i) & 1, abort_flag))) { ok = false; break; }
            tc_fence_after();
            uint32_t sr[TC_BN];
#pragma unroll
            for (int c = 0; c < TC_BN / 32; ++c)
                tmem_ld_32x32b_x32(tm_s + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
            tmem_ld_wait();
            const int k0 = j * TC_BN;
            // keys to mask in this tile (decided for the whole CTA): past the diagonal, padding of
            // this sequence, or older than some row's window
            const bool diag = k0 + TC_BN - 1 > len0 + q0;
            const bool pads = k0 < pe && k0 + TC_BN > ps;
            const bool old = window > 0 && k0 < len0 + q_end - window;
            if (pads || old) {
                // key e is visible iff (e <= lim, not padding, inside the window) or it is the query
                // itself: two intervals, before and after the padding, plus the query's own slot.
                // Branch-free (unsigned range tests): a short-circuit form diverges per element.
                const int lim = pos - k0;
                const int lo = window > 0 ? lim - window + 1 : -TC_BN;
                const int a1 = max(lo, 0), n1 = max(0, min(lim, ps - k0 - 1) - a1 + 1);
                const int a2 = max(lo, pe - k0), n2 = max(0, lim - a2 + 1);
#pragma unroll
                for (int e = 0; e < TC_BN; ++e) {
                    const bool vis = ((unsigned)(e - a1) < (unsigned)n1) | ((unsigned)(e - a2) < (unsigned)n2) | (e == lim);
                    sr[e] = vis ? sr[e] : __float_as_uint(-INFINITY);
                }
            } else if (diag) {  // only the causal diagonal: keys past the query's slot
                const int lim = pos - k0;
#pragma unroll
                for (int e = 0; e < TC_BN; ++e) sr[e] = e <= lim ? sr[e] : __float_as_uint(-INFINITY);
            }
            float mx = -INFINITY;  // three-input maxima: two scores per instruction
#pragma unroll
            for (int e = 0; e < TC_BN; e += 2) mx = fmax3(mx, __uint_as_float(sr[e]), __uint_as_float(sr[e + 1]));
            mx *= sl2;
            // lazy rescale, decided per row but executed by the whole warp (tcgen05.ld/st are warp-wide)
            const bool grow = mx > m_used + 8.0f;
            const float alpha = grow ? ex2_approx(m_used - mx) : 1.0f;
            if (i > 0 && __any_sync(0xffffffffu, grow)) {
                const bool w = confirm_pv(i);  // O must hold P V of the previous tile before it is scaled
                if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < DH / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(tm_o + c * 32, o);
                    tmem_ld_wait();
                    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float2 r2 = mul2(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), a2);
                        o[e] = __float_as_uint(r2.x);
                        o[e + 1] = __float_as_uint(r2.y);
                    }
                    tmem_st_32x32b_x32(tm_o + c * 32, o);
                }
                tmem_st_wait();
            }
            if (grow) {
                l *= alpha;
                m_used = mx;
            }
            // P = 2^(s * sl2 - m) as packed bf16 into the first 64 columns of this head's S region (a row
            // with no visible key yet keeps m = -inf and gets P = 0)
            const float nm = m_used == -INFINITY ? 0.f : -m_used;
            const float2 sl2x2 = make_float2(sl2, sl2), nmx2 = make_float2(nm, nm);
            float2 rs2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float2 x = fma2(make_float2(__uint_as_float(sr[half * 64 + 2 * e]),
                                                      __uint_as_float(sr[half * 64 + 2 * e + 1])),
                                          sl2x2, nmx2);
                    const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                    rs2 = add2(rs2, pp);
                    pk[e] = pack_bf16(pp.x, pp.y);
                }
                tmem_st_32x32b_x32(tm_s + half * 32, pk);
            }
            tmem_st_wait();
            l += rs2.x + rs2.y;
            // Observe the previous P V completion before releasing this P: o_done is then never more
            // than one phase ahead of this thread, so its parity waits stay unambiguous.
            if (i > 0) {
                const bool w = confirm_pv(i);
                if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
            }
            tc_fence_before();
            mbar_arrive(&p_full[r]);
        }
        // epilogue
        if (ok) ok = confirm_pv(nt);
        ok = __all_sync(0xffffffffu, ok);
        __nv_bfloat16* orow = out + (((size_t)b * T + t) * Hq + h0 + hh) * DH;
        if (ok && n_chunks == 1) {
            // O / l straight to the output
            tc_fence_after();
            const float inv = 1.f / l;
#pragma unroll 1
            for (int c = 0; c < DH / 32; ++c) {
                uint32_t o[32];
                tmem_ld_32x32b_x32(tm_o + c * 32, o);
                tmem_ld_wait();
                if (t < T) {
                    uint32_t wv[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        wv[e] = pack_bf16(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        reinterpret_cast<uint4*>(orow + c * 32)[v] =
                            make_uint4(wv[4 * v], wv[4 * v + 1], wv[4 * v + 2], wv[4 * v + 3]);
                }
            }
        } else if (n_chunks > 1) {
            // partial (unnormalised O, running max, sum) of this chunk; the last chunk to finish merges
            constexpr int REC = DH + 4;  // floats per (head, row) record, 16-byte multiple
            const int item = (b * (Hq / NH) + (int)blockIdx.y) * n_qt + qt;
            float* rec0 = ws + ((size_t)item * max_chunks * NH + hh) * TC_BM * REC + (size_t)row * REC;
            const size_t chunk_stride = (size_t)NH * TC_BM * REC;
            if (ok) {
                tc_fence_after();
                float* rec = rec0 + chunk * chunk_stride;
#pragma unroll 1
                for (int c = 0; c < DH / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(tm_o + c * 32, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        reinterpret_cast<float4*>(rec + c * 32)[v] =
                            make_float4(__uint_as_float(o[4 * v]), __uint_as_float(o[4 * v + 1]),
                                        __uint_as_float(o[4 * v + 2]), __uint_as_float(o[4 * v + 3]));
                }
                rec[DH] = m_used;
                rec[DH + 1] = l;
            }
            __threadfence();
            named_barrier(2, 128 * NH);
            if (threadIdx.x == 64) *merge_flag = ok && atomicAdd(&tickets[item], 1) == n_chunks - 1;
            named_barrier(2, 128 * NH);
            if (*merge_flag) {
                __threadfence();
                float M = -INFINITY;
                for (int c = 0; c < n_chunks; ++c) M = fmaxf(M, rec0[c * chunk_stride + DH]);
                float L = 0.f, acc[DH];
#pragma unroll
                for (int d = 0; d < DH; ++d) acc[d] = 0.f;
                for (int c = 0; c < n_chunks; ++c) {
                    const float* rc = rec0 + c * chunk_stride;
                    const float mc = rc[DH];
                    const float wgt = mc == -INFINITY ? 0.f : ex2_approx(mc - M);
                    L = fmaf(rc[DH + 1], wgt, L);
#pragma unroll
                    for (int v = 0; v < DH / 4; ++v) {
                        const float4 q4 = reinterpret_cast<const float4*>(rc)[v];
                        acc[4 * v] = fmaf(q4.x, wgt, acc[4 * v]);
                        acc[4 * v + 1] = fmaf(q4.y, wgt, acc[4 * v + 1]);
                        acc[4 * v + 2] = fmaf(q4.z, wgt, acc[4 * v + 2]);
                        acc[4 * v + 3] = fmaf(q4.w, wgt, acc[4 * v + 3]);
                    }
                }
                const float inv = 1.f / L;
                if (t < T) {
#pragma unroll
                    for (int v = 0; v < DH / 8; ++v)
                        reinterpret_cast<uint4*>(orow)[v] =
                            make_uint4(pack_bf16(acc[8 * v] * inv, acc[8 * v + 1] * inv),
                                       pack_bf16(acc[8 * v + 2] * inv, acc[8 * v + 3] * inv),
                                       pack_bf16(acc[8 * v + 4] * inv, acc[8 * v + 5] * inv),
                                       pack_bf16(acc[8 * v + 6] * inv, acc[8 * v + 7] * inv));
                }
                if (threadIdx.x == 64) tickets[item] = 0;  // ready for the next launch
            }
        }
    }
    if (!ok) {
        *abort_flag = 1;
        if (err) atomicOr(err, ERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Persistent form of the one-head-per-CTA kernel: grid = min(work items, SMs). Work items are
// (query tile, sequence, query head) triples, longest causal range first; CTA c takes items
// c, 2G-1-c, 2G+c, ... (a snake over the sorted list, so every CTA gets a similar total). Tensor
// memory, barriers and the TMA/MMA pipeline stay alive across items: the next item's Q and first
// scores load while the softmax warps finish the current item, whose output accumulator is then
// handed back to the MMA warp (o_free) before the next item's first PV overwrites it. Tiles are
// counted across items (g), so ring stages, score regions and barrier phases simply continue.
// Tensor memory holds three score regions and the output accumulator (4 x 128 columns): the scores
// run two tiles ahead of P V, so the scores a softmax pass needs are complete when it starts. With
// two regions the MMA thread could issue S of tile j+2 only after P V of tile j; since a thread that
// issues tcgen05.mma waits while the pipe is full, it then sat behind that S while P of tile j+1
// was already waiting, and the softmax warps waited for their next scores: about 2,100 cycles per
// tile against 1,024 of MMA work (clock64 timeline of one CTA, 0.6B 1x2048).
// ALT = false: one softmax warpgroup (warps 2-5); warp 0 streams the keys, warp 1 issues the score
// MMAs, warp 6 streams the values, warp 7 issues the P V MMAs.
// ALT = true, for long key ranges: two softmax warpgroups take alternate key tiles (warpgroup 1 the
// even global tile numbers, warpgroup 2 the odd ones), each thread a whole query row. With one
// warpgroup the softmax pass sets the period: about 1,400 cycles per tile of mostly dependent work on
// one warp per sub-partition, against 1,024 cycles of MMA work and 512 of exponentials. The two
// warpgroups keep each row's scale in step through shared memory: a tile's scale becomes final after
// the previous tile's (mbarrier fin, one per row quarter and tile parity); its exponentials start
// speculatively with the scale known so far and are recomputed in the rare tile where it moved.
// Each warpgroup sums its own tiles' probabilities at its own scale; the two sums meet at the end of
// the item, where each warpgroup writes half of the output columns. Warpgroup 0 holds the producers
// (warp 0 keys, 1 score MMAs, 2 values, 3 P V MMAs) and gives registers to the softmax warpgroups
// (setmaxnreg). The first two tiles of an item run without speculation and the second waits for the
// first, which costs more than the alternation saves on items of about 16 tiles or fewer (measured,
// shapes timed in both orders: 8B 1x32768 5.65 -> 5.21-5.25 ms, 8B 1x8192 0.391 -> 0.364 ms, 0.6B
// 8x4096 0.447 -> 0.472 ms, 0.6B 1x2048 20.3 -> 22.0 us).
template <bool ALT>
constexpr int ps_threads() { return ALT ? 128 + 256 : 64 + 128 + 64; }
constexpr int PS_KST = 3, PS_VST = 2;  // key and value ring stages
constexpr uint32_t PS_REG_PRODUCER = 56, PS_REG_SOFTMAX = 224;
// the split must fit the registers of the launch (168 per thread at 384 threads and one block per
// SM) and each sub-partition's register file (one producer warp and two softmax warps)
static_assert(4 * PS_REG_PRODUCER + 8 * PS_REG_SOFTMAX <= 12 * 168, "register split exceeds the launch");
static_assert(PS_REG_PRODUCER + 2 * PS_REG_SOFTMAX <= 512, "register split exceeds a sub-partition");
template <int DH, bool ALT>
struct PsLayout {
    static constexpr int NCH = DH / 64;
    static constexpr int Q_BYTES = TC_BM * DH * 2;
    static constexpr int KV_BYTES = TC_BN * DH * 2;
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_BYTES;
    static constexpr int V_OFF = K_OFF + PS_KST * KV_BYTES;
    static constexpr int BAR_OFF = V_OFF + PS_VST * KV_BYTES;
    // ALT: 37 barriers, then the row scales [2][128] and row sums [2][2][128] (floats). The other form
    // keeps the smaller size: the extra 3 KB move the shared-memory carve-out up a step, which cost it
    // 5-8% (0.6B 8x4096, 8B 1x8192).
    static constexpr int XCH_OFF = BAR_OFF + (ALT ? 512 : 256);
    static constexpr int SMEM = XCH_OFF + (ALT ? 6 * TC_BM * 4 : 0) + 1024;
};

template <int DH, bool SPEC, bool ALT>
__global__ void __launch_bounds__(ps_threads<ALT>(), 1)
    attn_prefill_persistent_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                                   const __grid_constant__ CUtensorMap tmV, int T, int Hq, int Hkv, int B,
                                   const int* __restrict__ len0p, const int* __restrict__ meta, int window, int ring,
                                   __nv_bfloat16* __restrict__ out, int* err) {
    using Ly = PsLayout<DH, ALT>;
    constexpr int NCH = Ly::NCH;
    constexpr uint32_t IDESC_S = idesc_bf16(TC_BM, TC_BN);
    constexpr uint32_t IDESC_O = idesc_bf16(TC_BM, DH, true);
    constexpr int NR = 3;                  // score regions in tensor memory
    constexpr uint32_t TM_O = NR * TC_BN;  // then the output accumulator: 512 columns in all
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Ly::BAR_OFF);
    uint64_t* q_full = bars;
    uint64_t* q_empty = bars + 1;
    uint64_t* k_full = bars + 2;   // [PS_KST]
    uint64_t* k_empty = bars + 5;  // [PS_KST]
    uint64_t* v_full = bars + 8;   // [PS_VST]
    uint64_t* v_empty = bars + 10; // [PS_VST]
    uint64_t* s_full = bars + 12;  // [NR] per score region
    uint64_t* p_full = bars + 15;  // [NR] per score region
    uint64_t* o_free = bars + 19;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 20);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 21);
    uint64_t* r_free = bars + 22;  // [NR] P V of the region's tile is done: the region can take new scores
    uint64_t* fin = bars + 25;     // ALT [4 row quarters][2 tile parities]: the tile's row scales are final
    uint64_t* l_meet = bars + 33;  // ALT [4 row quarters]: both warpgroups published the item's row sums

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_qt = (T + TC_BM - 1) / TC_BM;
    const int per_qt = B * Hq;
    const int n_items = n_qt * per_qt;
    const int G = (int)gridDim.x, c = (int)blockIdx.x;
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int i = 0; i < PS_KST; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < PS_VST; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < NR; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 128);  // the softmax warpgroup that owns the tile
            mbar_init(&r_free[i], 1);
        }
        mbar_init(o_free, ALT ? 256 : 128);
        if (ALT) {
            for (int i = 0; i < 8; ++i) mbar_init(&fin[i], 32);
            for (int i = 0; i < 4; ++i) mbar_init(&l_meet[i], 64);
        }
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;
    pdl_wait();  // Q and the cache come from the previous kernel
    pdl_trigger();
    const int len0 = *len0p;
    int ps_meta = 0, psh = 0;
    if (meta) {
        ps_meta = meta[0];
        psh = meta[1];
    }

    // The parameters of this CTA's round-th item (n_tiles = 0 when it has none left).
    struct Item {
        int b, h, q0, q_end, n_valid, j_lo, ja, jb, n_tiles, ps, pe;
    };
    auto item_of = [&](int round) -> Item {
        Item it{};
        const int k = round * G + ((round & 1) ? G - 1 - c : c);
        if (k >= n_items) return it;
        const int qt = n_qt - 1 - k / per_qt, rem = k % per_qt;
        it.b = rem / Hq;
        it.h = rem % Hq;
        it.q0 = qt * TC_BM;
        it.q_end = min(T, it.q0 + TC_BM);
        it.ps = ps_meta;
        it.pe = meta ? ps_meta + meta[kSeqMetaHead + it.b] : 0;
        it.n_valid = len0 + it.q_end;
        const int n_end = (it.n_valid + TC_BN - 1) / TC_BN;
        it.j_lo = window > 0 ? max(0, len0 + it.q0 - window + 1) / TC_BN : 0;
        it.ja = max(it.j_lo, (it.ps + TC_BN - 1) / TC_BN);
        it.jb = max(it.ja, min(it.pe / TC_BN, (len0 + it.q0) / TC_BN));
        it.n_tiles = n_end - it.j_lo - (it.jb - it.ja);
        return it;
    };
    auto tile_j = [](const Item& it, int i) { return it.j_lo + i < it.ja ? it.j_lo + i : it.j_lo + i + (it.jb - it.ja); };

    constexpr int W_VTMA = ALT ? 2 : 6, W_PV = ALT ? 3 : 7;
    const bool producer = ALT ? warp < 4 : (warp < 2 || warp >= 6);
    // with ALT the register split dominates each role's code, so that ptxas allocates it under the
    // new limit
    if (producer) {
        if constexpr (ALT) setmaxnreg_dec<PS_REG_PRODUCER>();
        if (warp == 0) {
            // ---------------- TMA producer
            if (lane == 0) {
                int g = 0;
                for (int round = 0; ok; ++round) {
                    const Item it = item_of(round);
                    if (it.n_tiles == 0) break;
                    const int jkv = it.h / (Hq / Hkv);
                    if (!mbar_wait_suspend(q_empty, (round & 1) ^ 1, abort_flag)) { ok = false; break; }
                    mbar_expect_tx(q_full, Ly::Q_BYTES);
                    for (int cc = 0; cc < NCH; ++cc)
                        tma_load_3d(smem + Ly::Q_OFF + cc * TC_BM * 128, &tmQ, q_full, cc * 64, it.q0, it.b * Hq + it.h);
                    for (int i = 0; i < it.n_tiles; ++i, ++g) {
                        const int s = g % PS_KST, j = tile_j(it, i);
                        const uint32_t free_ph = ((g / PS_KST) & 1) ^ 1;
                        const int y = ring ? (j * TC_BN) % ring : j * TC_BN;
                        const int z = (j * TC_BN < psh ? 0 : it.b) * Hkv + jkv;
                        if (!mbar_wait_suspend(&k_empty[s], free_ph, abort_flag)) { ok = false; break; }
                        mbar_expect_tx(&k_full[s], Ly::KV_BYTES);
                        for (int cc = 0; cc < NCH; ++cc)
                            tma_load_3d(smem + Ly::K_OFF + s * Ly::KV_BYTES + cc * TC_BN * 128, &tmK, &k_full[s], cc * 64, y, z);
                    }
                }
            }
        } else if (warp == W_VTMA) {
            // ---------------- TMA producer for the value tiles, a warp of its own: a key stage is freed by
            // its scores, a value stage by its P V, two tiles apart, so one in-order producer would hold
            // back the keys of the scores that run ahead
            if (lane == 0) {
                int g = 0;
                for (int round = 0; ok; ++round) {
                    const Item it = item_of(round);
                    if (it.n_tiles == 0) break;
                    const int jkv = it.h / (Hq / Hkv);
                    for (int i = 0; i < it.n_tiles; ++i, ++g) {
                        const int s = g & 1, j = tile_j(it, i);
                        const uint32_t free_ph = ((g >> 1) & 1) ^ 1;
                        const int y = ring ? (j * TC_BN) % ring : j * TC_BN;
                        const int z = (j * TC_BN < psh ? 0 : it.b) * Hkv + jkv;
                        if (!mbar_wait_suspend(&v_empty[s], free_ph, abort_flag)) { ok = false; break; }
                        mbar_expect_tx(&v_full[s], Ly::KV_BYTES);
                        for (int cc = 0; cc < NCH; ++cc)
                            tma_load_3d(smem + Ly::V_OFF + s * Ly::KV_BYTES + cc * TC_BN * 128, &tmV, &v_full[s], cc * 64, y, z);
                    }
                }
            }
        } else if (warp == 1) {
            // ---------------- score MMAs: S of tile gi (key stage gi % PS_KST) into region gi % NR, once
            // P V of tile gi - NR (issued by the P V warp) has finished reading that region. A thread issuing
            // tcgen05.mma waits while the pipe is full, so the score and the P V batches come from two
            // threads: while one waits with its batch, the other's work keeps the pipe fed.
            if (lane == 0) {
                int g = 0;  // tiles of earlier items
                for (int round = 0; ok; ++round) {
                    const Item it = item_of(round);
                    const int nt = it.n_tiles;
                    if (nt == 0) break;
                    if (!mbar_wait_suspend(q_full, round & 1, abort_flag)) { ok = false; break; }
                    for (int i = 0; i < nt; ++i) {
                        const int gi = g + i, s = gi % PS_KST, r = gi % NR;
                        if (!mbar_wait_suspend(&k_full[s], (gi / PS_KST) & 1, abort_flag)) { ok = false; break; }
                        // region r's next completion would be P V of tile gi itself, not yet possible: the
                        // parity wait cannot alias
                        if (gi >= NR && !mbar_wait_suspend(&r_free[r], ((gi - NR) / NR) & 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sq = smem_u32(smem + Ly::Q_OFF);
                        const uint32_t sk = smem_u32(smem + Ly::K_OFF + s * Ly::KV_BYTES);
#pragma unroll
                        for (int kk = 0; kk < DH / 16; ++kk) {
                            const uint32_t off = (kk >> 2) * TC_BM * 128 + (kk & 3) * 32;
                            umma_bf16_ss(tmem + r * TC_BN, sdesc_kmajor_sw128(sq + off), sdesc_kmajor_sw128(sk + off),
                                         IDESC_S, kk > 0);
                        }
                        umma_commit(&s_full[r]);
                        umma_commit(&k_empty[s]);
                        if (i == nt - 1) umma_commit(q_empty);  // the item's last score releases Q
                    }
                    g += nt;
                }
            }
        } else if (warp == W_PV) {
            // ---------------- P V MMAs: O += P V of tile gi, P read from region gi % NR (A operand in
            // tensor memory), V from value stage gi & 1
            int g = 0;
            for (int round = 0; ok; ++round) {
                const Item it = item_of(round);
                const int nt = it.n_tiles;
                if (nt == 0) break;
                for (int i = 0; ok && i < nt; ++i) {
                    const int gi = g + i, s = gi & 1, r = gi % NR;
                    const int j = tile_j(it, i);
                    if (!__all_sync(0xffffffffu, mbar_wait_suspend(&v_full[s], (gi >> 1) & 1, abort_flag))) { ok = false; break; }
                    uint8_t* sv = smem + Ly::V_OFF + s * Ly::KV_BYTES;
                    const int r0 = it.n_valid - j * TC_BN;  // first stale key row of this tile
                    if (r0 < TC_BN) {
                        for (int e = lane; e < (TC_BN - r0) * 8 * NCH; e += 32) {
                            const int cc = e / ((TC_BN - r0) * 8), rem = e % ((TC_BN - r0) * 8);
                            reinterpret_cast<uint4*>(sv + cc * TC_BN * 128 + (r0 + rem / 8) * 128)[rem % 8] =
                                make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                    }
                    __syncwarp();
                    if (lane == 0) {
                        bool w = i > 0 || mbar_wait_suspend(o_free, (round & 1) ^ 1, abort_flag);  // previous item's O read out
                        w = w && mbar_wait_suspend(&p_full[r], (gi / NR) & 1, abort_flag);
                        if (w) {
                            tc_fence_after();
                            const uint32_t svv = smem_u32(sv);
#pragma unroll
                            for (int kk = 0; kk < TC_BN / 16; ++kk) {
                                const uint64_t bd = sdesc_mnmajor_sw128(svv + kk * 16 * 128, TC_BN * 128);
                                umma_bf16_ts(tmem + TM_O, tmem + r * TC_BN + kk * 8, bd, IDESC_O, (i | kk) != 0);
                            }
                            umma_commit(&v_empty[s]);
                            umma_commit(&r_free[r]);
                        }
                        ok = w;
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                }
                g += nt;
            }
        }
    } else if constexpr (ALT) {
        setmaxnreg_inc<PS_REG_SOFTMAX>();
        // ---------------- softmax warpgroups: thread <-> query row (TMEM lane); warpgroup wg takes the
        // tiles whose global number has parity wg
        const int wg = (warp >> 2) - 1;
        const int quarter = warp & 3, row = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tm_o = tmem + lane_off + TM_O;
        const float sl2 = kLog2e / sqrtf((float)DH);
        volatile float* m_sh = reinterpret_cast<volatile float*>(smem + Ly::XCH_OFF);  // [item parity][row]
        volatile float* l_sh = m_sh + 2 * TC_BM;  // [item parity][warpgroup][row]
        // P V of global tile k (and so every earlier one) has completed. The region's next completion
        // would be P V of tile k + NR, which needs a P of this warpgroup that is not released yet
        // (k + NR has the parity of the caller's tile k + 1), so the parity wait cannot alias.
        auto pv_done = [&](int k) -> bool { return mbar_wait_suspend(&r_free[k % NR], (k / NR) & 1, abort_flag); };
        // The row scales of global tile k are final. Barrier fin[quarter][k & 1] completes one phase
        // per tile of that parity; its next phase needs tile k + 2, which waits for the caller's tile
        // k + 1 to be final, so the parity wait cannot alias.
        auto fin_wait = [&](int k) -> bool {
            return mbar_wait_suspend(&fin[quarter * 2 + (k & 1)], (k >> 1) & 1, abort_flag);
        };
        int g = 0;
        for (int round = 0; ok; ++round) {
            const Item it = item_of(round);
            const int nt = it.n_tiles;
            if (nt == 0) break;
            const int t = it.q0 + row, pos = len0 + t;
            volatile float* m_row = m_sh + (round & 1) * TC_BM + row;
            float m_l = -INFINITY, l = 0.f;  // this warpgroup's share of the row sum, at scale m_l
            for (int i = ((g & 1) == wg) ? 0 : 1; i < nt; i += 2) {
                const int gi = g + i, r = gi % NR;
                const int j = tile_j(it, i);
                const uint32_t tm_s = tmem + lane_off + r * TC_BN;
                if (!__all_sync(0xffffffffu, mbar_wait_suspend(&s_full[r], (gi / NR) & 1, abort_flag))) { ok = false; break; }
                tc_fence_after();
                uint32_t sr[TC_BN];
#pragma unroll
                for (int cc = 0; cc < TC_BN / 32; ++cc)
                    tmem_ld_32x32b_x32(tm_s + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[cc * 32]));
                tmem_ld_wait();
                const int k0 = j * TC_BN;
                const bool diag = k0 + TC_BN - 1 > len0 + it.q0;
                const bool pads = k0 < it.pe && k0 + TC_BN > it.ps;
                const bool old = window > 0 && k0 < len0 + it.q_end - window;
                if (pads || old) {
                    // visible: (i <= lim, not padding, inside the window) or the query itself; branch-free
                    const int lim = pos - k0;
                    const int lo = window > 0 ? lim - window + 1 : -TC_BN;
                    const int a1 = max(lo, 0), n1 = max(0, min(lim, it.ps - k0 - 1) - a1 + 1);
                    const int a2 = max(lo, it.pe - k0), n2 = max(0, lim - a2 + 1);
#pragma unroll
                    for (int e = 0; e < TC_BN; ++e) {
                        const bool vis =
                            ((unsigned)(e - a1) < (unsigned)n1) | ((unsigned)(e - a2) < (unsigned)n2) | (e == lim);
                        sr[e] = vis ? sr[e] : __float_as_uint(-INFINITY);
                    }
                } else if (diag) {
                    const int lim = pos - k0;
#pragma unroll
                    for (int e = 0; e < TC_BN; ++e) sr[e] = e <= lim ? sr[e] : __float_as_uint(-INFINITY);
                }
                // P = 2^(s * sl2 - m) as packed bf16 into the first 64 columns of this tile's region (a row
                // with no visible key yet keeps m = -inf and gets P = 0); rs2 = their row sum
                auto exps = [&](float mref, float2& rs2) {
                    const float nm = mref == -INFINITY ? 0.f : -mref;
                    const float2 sl2x2 = make_float2(sl2, sl2), nmx2 = make_float2(nm, nm);
                    rs2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t pk[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const float2 x = fma2(make_float2(__uint_as_float(sr[half * 64 + 2 * e]),
                                                              __uint_as_float(sr[half * 64 + 2 * e + 1])),
                                                  sl2x2, nmx2);
                            const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                            rs2 = add2(rs2, pp);
                            pk[e] = pack_bf16(pp.x, pp.y);
                        }
                        tmem_st_32x32b_x32(tm_s + half * 32, pk);
                    }
                };
                // SPEC: the exponentials start with the scale published after this warpgroup's previous
                // tile of the item (or later) while the tile maximum is reduced beside them; they are
                // recomputed when the final scale differs. Decisions are warp-uniform (tcgen05.st is
                // warp-wide).
                const float m_ref = i >= 2 ? *m_row : -INFINITY;
                float2 rs2;
                const bool spec = SPEC && __all_sync(0xffffffffu, m_ref != -INFINITY);
                if (spec) exps(m_ref, rs2);
                float mx = -INFINITY;
                if constexpr (SPEC) {
                    float m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
                    for (int e = 0; e < TC_BN; e += 8) {
                        mx = fmax3(mx, __uint_as_float(sr[e]), __uint_as_float(sr[e + 1]));
                        m1 = fmax3(m1, __uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3]));
                        m2 = fmax3(m2, __uint_as_float(sr[e + 4]), __uint_as_float(sr[e + 5]));
                        m3 = fmax3(m3, __uint_as_float(sr[e + 6]), __uint_as_float(sr[e + 7]));
                    }
                    mx = fmaxf(fmaxf(mx, m1), fmaxf(m2, m3));
                } else {
#pragma unroll
                    for (int e = 0; e < TC_BN; e += 2) mx = fmax3(mx, __uint_as_float(sr[e]), __uint_as_float(sr[e + 1]));
                }
                mx *= sl2;
                // the scale after the previous tile of the item (final once that tile is)
                if (i > 0 && !__all_sync(0xffffffffu, fin_wait(gi - 1))) { ok = false; break; }
                const float m_prev = i > 0 ? *m_row : -INFINITY;
                // lazy rescale, decided per row but executed by the whole warp
                const bool grow = mx > m_prev + 8.0f;
                const float m_new = grow ? mx : m_prev;
                if (i > 0 && __any_sync(0xffffffffu, grow)) {
                    // O holds P V of every earlier tile at scale m_prev
                    const bool w = pv_done(gi - 1);
                    if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                    tc_fence_after();
                    const float alpha = grow ? ex2_approx(m_prev - mx) : 1.0f;
                    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll 1
                    for (int cc = 0; cc < DH / 32; ++cc) {
                        uint32_t o[32];
                        tmem_ld_32x32b_x32(tm_o + cc * 32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float2 r2 = mul2(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), a2);
                            o[e] = __float_as_uint(r2.x);
                            o[e + 1] = __float_as_uint(r2.y);
                        }
                        tmem_st_32x32b_x32(tm_o + cc * 32, o);
                    }
                    tmem_st_wait();
                }
                if (!spec || __any_sync(0xffffffffu, m_new != m_ref)) {
                    if (spec) tmem_st_wait();  // the speculative P is overwritten
                    exps(m_new, rs2);
                }
                // this warpgroup's share of the row sum moves to the new scale (m_new > m_l, so finite)
                if (m_new != m_l) {
                    l *= ex2_approx(m_l - m_new);
                    m_l = m_new;
                }
                tmem_st_wait();
                l += rs2.x + rs2.y;
                *m_row = m_new;
                tc_fence_before();
                mbar_arrive(&p_full[r]);
                mbar_arrive(&fin[quarter * 2 + (gi & 1)]);  // releases the scale written above
            }
            if (!ok) break;
            // the item's last tile is final: the row's final scale, and once its P V is done, O. Both
            // waits come before the meeting, which neither warpgroup passes before both arrive, so no
            // tile of the next item (whose P V would complete the region barrier's next phase) can run
            // before both waits are over.
            const int last = g + nt - 1;
            ok = __all_sync(0xffffffffu, fin_wait(last) && pv_done(last));
            if (!ok) break;
            const float m_fin = *m_row;
            volatile float* l_row = l_sh + (round & 1) * 2 * TC_BM + row;
            l_row[wg * TC_BM] = m_l == m_fin ? l : l * ex2_approx(m_l - m_fin);
            mbar_arrive(&l_meet[quarter]);
            ok = __all_sync(0xffffffffu, mbar_wait_suspend(&l_meet[quarter], round & 1, abort_flag));
            if (!ok) break;
            // O / l to the output, this warpgroup's half of the columns, then hand the accumulator back
            tc_fence_after();
            const float inv = 1.f / (l_row[0] + l_row[TC_BM]);
            __nv_bfloat16* orow = out + (((size_t)it.b * T + t) * Hq + it.h) * DH + wg * (DH / 2);
#pragma unroll 1
            for (int cc = 0; cc < DH / 64; ++cc) {
                uint32_t o[32];
                tmem_ld_32x32b_x32(tm_o + wg * (DH / 2) + cc * 32, o);
                tmem_ld_wait();
                if (t < T) {
                    uint32_t wv[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        wv[e] = pack_bf16(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        reinterpret_cast<uint4*>(orow + cc * 32)[v] =
                            make_uint4(wv[4 * v], wv[4 * v + 1], wv[4 * v + 2], wv[4 * v + 3]);
                }
            }
            tc_fence_before();
            mbar_arrive(o_free);
            g += nt;
        }
    } else {
        // ---------------- softmax warps: thread <-> query row (TMEM lane)
        const int quarter = warp & 3, row = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tm_o = tmem + lane_off + TM_O;
        const float sl2 = kLog2e / sqrtf((float)DH);
        // P V of global tile k (and so every earlier one) has completed. The region's next completion
        // would be P V of tile k + NR, which needs a P this thread has not released yet, so the parity
        // wait cannot alias; P is therefore released without waiting for the previous P V.
        auto pv_done = [&](int k) -> bool { return mbar_wait_suspend(&r_free[k % NR], (k / NR) & 1, abort_flag); };
        int g = 0;
        for (int round = 0; ok; ++round) {
            const Item it = item_of(round);
            const int nt = it.n_tiles;
            if (nt == 0) break;
            const int t = it.q0 + row, pos = len0 + t;
            float m_used = -INFINITY, l = 0.f;
            for (int i = 0; i < nt; ++i) {
                const int gi = g + i, r = gi % NR;
                const int j = tile_j(it, i);
                const uint32_t tm_s = tmem + lane_off + r * TC_BN;
                if (!__all_sync(0xffffffffu, mbar_wait_suspend(&s_full[r], (gi / NR) & 1, abort_flag))) { ok = false; break; }
                tc_fence_after();
                uint32_t sr[TC_BN];
#pragma unroll
                for (int cc = 0; cc < TC_BN / 32; ++cc)
                    tmem_ld_32x32b_x32(tm_s + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[cc * 32]));
                tmem_ld_wait();
                const int k0 = j * TC_BN;
                const bool diag = k0 + TC_BN - 1 > len0 + it.q0;
                const bool pads = k0 < it.pe && k0 + TC_BN > it.ps;
                const bool old = window > 0 && k0 < len0 + it.q_end - window;
                if (pads || old) {
                    // visible: (i <= lim, not padding, inside the window) or the query itself; branch-free
                    const int lim = pos - k0;
                    const int lo = window > 0 ? lim - window + 1 : -TC_BN;
                    const int a1 = max(lo, 0), n1 = max(0, min(lim, it.ps - k0 - 1) - a1 + 1);
                    const int a2 = max(lo, it.pe - k0), n2 = max(0, lim - a2 + 1);
#pragma unroll
                    for (int e = 0; e < TC_BN; ++e) {
                        const bool vis =
                            ((unsigned)(e - a1) < (unsigned)n1) | ((unsigned)(e - a2) < (unsigned)n2) | (e == lim);
                        sr[e] = vis ? sr[e] : __float_as_uint(-INFINITY);
                    }
                } else if (diag) {
                    const int lim = pos - k0;
#pragma unroll
                    for (int e = 0; e < TC_BN; ++e) sr[e] = e <= lim ? sr[e] : __float_as_uint(-INFINITY);
                }
                // P = 2^(s * sl2 - m) as packed bf16 into the first 64 columns of this tile's region (a row
                // with no visible key yet keeps m = -inf and gets P = 0); rs2 = their row sum
                auto exps = [&](float mref, float2& rs2) {
                    const float nm = mref == -INFINITY ? 0.f : -mref;
                    const float2 sl2x2 = make_float2(sl2, sl2), nmx2 = make_float2(nm, nm);
                    rs2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t pk[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const float2 x = fma2(make_float2(__uint_as_float(sr[half * 64 + 2 * e]),
                                                              __uint_as_float(sr[half * 64 + 2 * e + 1])),
                                                  sl2x2, nmx2);
                            const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                            rs2 = add2(rs2, pp);
                            pk[e] = pack_bf16(pp.x, pp.y);
                        }
                        tmem_st_32x32b_x32(tm_s + half * 32, pk);
                    }
                };
                // SPEC: the exponentials start with the running maximum while the tile maximum is reduced
                // beside them (lazy rescaling keeps m_used in most tiles); a warp recomputes them when one
                // of its rows grew. The decision is warp-uniform: exps() issues tcgen05.st, which every
                // lane of the warp must execute.
                float2 rs2;
                const bool spec = SPEC && __all_sync(0xffffffffu, m_used != -INFINITY);
                if (spec) exps(m_used, rs2);
                // three-input maxima, two scores per instruction; beside the speculative exponentials the
                // reduction runs as four independent chains so that it finishes with them
                float mx = -INFINITY;
                if constexpr (SPEC) {
                    float m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
                    for (int e = 0; e < TC_BN; e += 8) {
                        mx = fmax3(mx, __uint_as_float(sr[e]), __uint_as_float(sr[e + 1]));
                        m1 = fmax3(m1, __uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3]));
                        m2 = fmax3(m2, __uint_as_float(sr[e + 4]), __uint_as_float(sr[e + 5]));
                        m3 = fmax3(m3, __uint_as_float(sr[e + 6]), __uint_as_float(sr[e + 7]));
                    }
                    mx = fmaxf(fmaxf(mx, m1), fmaxf(m2, m3));
                } else {
#pragma unroll
                    for (int e = 0; e < TC_BN; e += 2) mx = fmax3(mx, __uint_as_float(sr[e]), __uint_as_float(sr[e + 1]));
                }
                mx *= sl2;
                const bool grow = mx > m_used + 8.0f;
                const float alpha = grow ? ex2_approx(m_used - mx) : 1.0f;
                if (i > 0 && __any_sync(0xffffffffu, grow)) {
                    const bool w = pv_done(gi - 1);  // O must hold P V of the previous tile before it is scaled
                    if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll 1
                    for (int cc = 0; cc < DH / 32; ++cc) {
                        uint32_t o[32];
                        tmem_ld_32x32b_x32(tm_o + cc * 32, o);
                        tmem_ld_wait();
                        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float2 r2 = mul2(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), a2);
                            o[e] = __float_as_uint(r2.x);
                            o[e + 1] = __float_as_uint(r2.y);
                        }
                        tmem_st_32x32b_x32(tm_o + cc * 32, o);
                    }
                    tmem_st_wait();
                }
                if (grow) {
                    l *= alpha;
                    m_used = mx;
                }
                if (!spec || __any_sync(0xffffffffu, grow)) {
                    if (spec) tmem_st_wait();  // the speculative P is overwritten
                    exps(m_used, rs2);
                }
                tmem_st_wait();
                l += rs2.x + rs2.y;
                tc_fence_before();
                mbar_arrive(&p_full[r]);
            }
            if (ok) ok = pv_done(g + nt - 1);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            // O / l to the output, then hand the accumulator back to the MMA warp
            tc_fence_after();
            __nv_bfloat16* orow = out + (((size_t)it.b * T + t) * Hq + it.h) * DH;
            const float inv = 1.f / l;
#pragma unroll 1
            for (int cc = 0; cc < DH / 32; ++cc) {
                uint32_t o[32];
                tmem_ld_32x32b_x32(tm_o + cc * 32, o);
                tmem_ld_wait();
                if (t < T) {
                    uint32_t wv[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        wv[e] = pack_bf16(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        reinterpret_cast<uint4*>(orow + cc * 32)[v] =
                            make_uint4(wv[4 * v], wv[4 * v + 1], wv[4 * v + 2], wv[4 * v + 3]);
                }
            }
            tc_fence_before();
            mbar_arrive(o_free);
            g += nt;
        }
    }
    if (!ok) {
        *abort_flag = 1;
        if (err) atomicOr(err, ERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}


// ------------------------------------------------------------------------------------- decode
// Keys per decode CTA: long chunks amortise each CTA's fixed work over long caches, shorter ones keep
// more CTAs busy on short caches; a rolling buffer uses the shortest so that its ring (a multiple of
// 256) never wraps inside a chunk.
constexpr int DEC_CHUNK = 1024, DEC_CHUNK_SHORT = 512, DEC_CHUNK_RING = 256;
// Four compute warps and one TMA warp. The TMA warp streams the chunk's key tiles, then its value
// tiles (128 cache rows each, 128-byte swizzle) through two or three shared-memory stages; the compute warps
// run the two small contractions on the tensor cores with warp-level mma (m16n8k16, bf16 in, fp32
// accumulate): scores S^T = K q^T with the chunk's keys as rows and the group's query heads as the
// 8 columns, and O^T += V^T P^T with head_dim as rows. That leaves the CUDA cores only the softmax of
// G x CH scores, so the kernel streams K and V at HBM speed for any group size. Its waits park the
// thread with a suspend hint, as in every tcgen05 kernel here (0.6B 64 @ 4096 decode step 5.47 -> 5.40 ms).
constexpr int DEC_WARPS = 4, DEC_THREADS = 32 * (DEC_WARPS + 1), DEC_TK = 128;

template <int DH, int G, int CH>
struct DecLayout {
    static constexpr int NCH = DH / 64;                  // 64-column boxes per cache row
    static constexpr int STAGE = DEC_TK * DH * 2;        // bytes per stage: 32 KB (dh 128) / 16 KB (dh 64)
    static constexpr int NS = DH >= 128 ? 2 : 3;         // stages: two CTAs fit an SM
    // scores / probabilities [G][CH], later reused for the cross-warp sums [warps][G][DH]
    static constexpr int SBUF = G * CH > DEC_WARPS * G * DH ? G * CH : DEC_WARPS * G * DH;
    static constexpr int SBUF_OFF = NS * STAGE;
    static constexpr int BAR_OFF = SBUF_OFF + SBUF * 4;
    static constexpr int SMEM = BAR_OFF + 2 * NS * 8 + 16 + 1024;  // + alignment slack
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
// D (16x8 fp32) += A (16x16 bf16, row-major) B (16x8 bf16, column-major), one warp
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Shared address of the 16-byte chunk `dc` (8 columns) of row `row` in a stage of NCH boxes of
// 128 rows x 128 bytes written by TMA with the 128-byte swizzle (box base 1024-byte aligned).
template <int NCH>
__device__ __forceinline__ uint32_t swz_addr(uint32_t stage, int row, int dc) {
    return stage + (uint32_t)((dc >> 3) * DEC_TK * 128 + row * 128 + (((dc & 7) ^ (row & 7)) << 4));
}

// Workspace layout per (b, q-head, split): [m, l] floats, then DH floats of unnormalised output.
// A CTA owns CH keys of one (sequence, kv head) and serves all G query heads of that group from one
// read of K and V.
template <int DH, int G, int CH>
__global__ void __launch_bounds__(DEC_THREADS)
    attn_decode_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                             const __nv_bfloat16* __restrict__ q, int Hq, int Hkv, const int* __restrict__ len0p,
                             const int* __restrict__ meta, int window, int ring, float* __restrict__ work, int* err) {
    static_assert(G <= 8, "the query heads of a group are the 8 columns of the mma");
    using Ly = DecLayout<DH, G, CH>;
    constexpr int NCH = Ly::NCH;
    constexpr int MT = DEC_TK / 16 / DEC_WARPS;  // 16-key tiles per warp and stage
    constexpr int REC = DH + 2;
    extern __shared__ uint8_t dsm_raw[];
    const uint32_t raw_addr = smem_u32(dsm_raw);
    uint8_t* dsm = dsm_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    float* sbuf = reinterpret_cast<float*>(dsm + Ly::SBUF_OFF);
    uint64_t* full = reinterpret_cast<uint64_t*>(dsm + Ly::BAR_OFF);
    uint64_t* empty = full + Ly::NS;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + Ly::NS);
    __shared__ float stat[G][2];
    auto sc = reinterpret_cast<float(*)[CH]>(sbuf);
    auto red = reinterpret_cast<float(*)[G][DH]>(sbuf);

    pdl_wait();
    pdl_trigger();
    const int split = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
    const int nsplit = gridDim.x;
    const int n = *len0p + 1;
    // keys [lo, n): a sliding window keeps the last `window`; chunks are aligned to CH slots
    const int lo = window > 0 ? max(0, n - window) : 0;
    const int s0 = lo / CH * CH + split * CH, s1 = min(n, s0 + CH);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, tq = lane & 3;  // mma fragment coordinates: group (row / column) and thread in group
    float* wb = work + (((size_t)b * Hq + (size_t)j * G) * nsplit + split) * REC;
    // padding slots [ps, pe) of this sequence; slots below psh (a multiple of 128) live in sequence 0;
    // a rolling buffer stores slot s at s mod ring (ring a multiple of CH, so a chunk stays contiguous)
    int ps = 0, pe = 0, psh = 0;
    if (meta) {
        ps = meta[0];
        psh = meta[1];
        pe = ps + meta[kSeqMetaHead + b];
    }
    if (s0 >= n) return;  // past the length: the merge does not read this chunk's records
    if (s0 >= ps && s1 <= pe) {  // only padding: a record of weight 0 (its output floats are not read)
        if (threadIdx.x < G) {
            wb[(size_t)threadIdx.x * nsplit * REC + 0] = -INFINITY;
            wb[(size_t)threadIdx.x * nsplit * REC + 1] = 0.f;
        }
        return;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < Ly::NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], DEC_WARPS);
        }
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    __syncthreads();
    const int nt = (s1 - s0 + DEC_TK - 1) / DEC_TK;  // stages per pass
    bool ok = true;

    if (warp == DEC_WARPS) {
        // ---------------- TMA warp: key tiles 0..nt-1, then value tiles (rows past the cache read as zero)
        if (lane == 0) {
            for (int it = 0; it < 2 * nt; ++it) {
                const int pass = it >= nt, t = it - pass * nt, stg = it % Ly::NS;
                if (it >= Ly::NS && !mbar_wait_suspend(&empty[stg], ((it / Ly::NS) - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const int a = s0 + t * DEC_TK;
                const int y = ring ? a % ring : a;
                const int z = (a < psh ? 0 : b) * Hkv + j;
                uint8_t* dst = dsm + stg * Ly::STAGE;
                mbar_expect_tx(&full[stg], Ly::STAGE);
                for (int cc = 0; cc < NCH; ++cc)
                    tma_load_3d(dst + cc * DEC_TK * 128, pass ? &tmV : &tmK, &full[stg], cc * 64, y, z);
            }
            if (!ok) {
                *abort_flag = 1;
                if (err) atomicOr(err, ERR_TIMEOUT);
            }
        }
        return;  // the compute warps wait for every stage it issued before they finish
    }

    // ---------------- compute warps (named barrier 1 spans these 128 threads only)
    const float sl2 = kLog2e / sqrtf((float)DH);
    // B fragments of q^T: column gq = query head gq of the group, rows = head_dim (zero columns past G)
    uint32_t qf[DH / 16][2];
    {
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(q + ((size_t)b * Hq + (size_t)j * G + gq) * DH);
#pragma unroll
        for (int ks = 0; ks < DH / 16; ++ks) {
            qf[ks][0] = gq < G ? qrow[ks * 8 + tq] : 0u;
            qf[ks][1] = gq < G ? qrow[ks * 8 + 4 + tq] : 0u;
        }
    }
    auto wait_full = [&](int it) -> bool {
        return __all_sync(0xffffffffu, mbar_wait_suspend(&full[it % Ly::NS], (it / Ly::NS) & 1, abort_flag));
    };
    auto release = [&](int it) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[it % Ly::NS]);
    };
    // pass 1: scores S^T (keys x heads), in log2 units
    for (int t = 0; t < nt && ok; ++t) {
        if (!wait_full(t)) {
            ok = false;
            break;
        }
        const uint32_t stage = smem_u32(dsm + (t % Ly::NS) * Ly::STAGE);
        const int a = s0 + t * DEC_TK;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const int kb = (m * DEC_WARPS + warp) * 16;  // first key of this 16-key tile within the stage
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            const int lrow = kb + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int ks = 0; ks < DH / 16; ++ks) {
                uint32_t af[4];
                ldsm_x4(swz_addr<NCH>(stage, lrow, 2 * ks + (lane >> 4)), af);
                mma_16816(d, af, qf[ks][0], qf[ks][1]);
            }
            // d[0], d[1]: key kb + gq, heads 2tq, 2tq+1; d[2], d[3]: key kb + gq + 8
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int s = a + kb + gq + 8 * r;
                if (s < s1) {
                    const bool vis = s >= lo && (s < ps || s >= pe);  // outside the window, or padding
#pragma unroll
                    for (int c = 0; c < 2; ++c)
                        if (2 * tq + c < G) sc[2 * tq + c][s - s0] = vis ? d[2 * r + c] * sl2 : -INFINITY;
                }
            }
        }
        release(t);
    }
    named_barrier(1, 32 * DEC_WARPS);
    // chunk max and exponentials, one warp per head
    const int cnt = s1 - s0;
    for (int h = warp; h < G; h += DEC_WARPS) {
        float mx = -INFINITY;
        for (int i = lane; i < cnt; i += 32) mx = fmaxf(mx, sc[h][i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float sum = 0.f;
        for (int i = lane; i < cnt; i += 32) {
            const float e = mx == -INFINITY ? 0.f : exp2f(sc[h][i] - mx);  // a chunk with no visible key
            sc[h][i] = e;
            sum += e;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) {
            stat[h][0] = mx;
            stat[h][1] = sum;
        }
    }
    named_barrier(1, 32 * DEC_WARPS);
    // pass 2: O^T (head_dim x heads) += V^T P^T, P rounded to bf16 for the mma
    float o[DH / 16][4];
#pragma unroll
    for (int mt = 0; mt < DH / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    auto prob = [&](int s) -> float { return (gq < G && s < s1) ? sc[gq][s - s0] : 0.f; };
    for (int t = 0; t < nt && ok; ++t) {
        if (!wait_full(nt + t)) {
            ok = false;
            break;
        }
        uint8_t* stage_p = dsm + ((nt + t) % Ly::NS) * Ly::STAGE;
        const uint32_t stage = smem_u32(stage_p);
        const int a = s0 + t * DEC_TK;
        if (a + DEC_TK > s1) {
            // value rows past the last key hold stale cache contents: zero this warp's, so that
            // 0 * NaN cannot reach O
            for (int m = 0; m < MT; ++m) {
                const int kb = (m * DEC_WARPS + warp) * 16;
                for (int e = lane; e < 16 * NCH * 8; e += 32) {
                    const int row = kb + e / (NCH * 8), dc = e % (NCH * 8);
                    if (a + row >= s1)
                        *reinterpret_cast<uint4*>(stage_p + (swz_addr<NCH>(stage, row, dc) - stage)) =
                            make_uint4(0, 0, 0, 0);
                }
            }
            __syncwarp();
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const int kb = (m * DEC_WARPS + warp) * 16;
            const int s = a + kb + 2 * tq;
            const uint32_t b0 = pack_bf16(prob(s), prob(s + 1)), b1 = pack_bf16(prob(s + 8), prob(s + 9));
            const int vrow = kb + (lane & 7) + ((lane >> 4) & 1) * 8;  // key row of this lane's address
#pragma unroll
            for (int mt = 0; mt < DH / 16; ++mt) {
                uint32_t af[4];
                ldsm_x4_trans(swz_addr<NCH>(stage, vrow, 2 * mt + ((lane >> 3) & 1)), af);
                mma_16816(o[mt], af, b0, b1);
            }
        }
        if (a + DEC_TK > s1) fence_proxy_async_smem();  // the zeroing stores precede the next TMA write
        release(nt + t);
    }
    if (!ok) {
        *abort_flag = 1;
        if (err) atomicOr(err, ERR_TIMEOUT);
    }
    named_barrier(1, 32 * DEC_WARPS);  // every warp is done with the probabilities before their space is reused
    // o[mt]: rows (head_dim) mt*16 + gq (+8), columns (heads) 2tq, 2tq+1
#pragma unroll
    for (int mt = 0; mt < DH / 16; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int c = 0; c < 2; ++c)
                if (2 * tq + c < G) red[warp][2 * tq + c][mt * 16 + gq + 8 * r] = o[mt][2 * r + c];
    named_barrier(1, 32 * DEC_WARPS);
    for (int i = threadIdx.x; i < G * DH; i += 32 * DEC_WARPS) {
        const int h = i / DH, dd = i % DH;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < DEC_WARPS; ++w) v += red[w][h][dd];
        float* rec = wb + (size_t)h * nsplit * REC;
        rec[2 + dd] = v;
        if (dd == 0) {
            rec[0] = stat[h][0];
            rec[1] = stat[h][1];
        }
    }
}

// Merge the chunks of one (b, q-head) by log-sum-exp: O = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i.
// Only chunks that can hold keys of this call are read (chunks [lo / CH, (n - 1) / CH] of the
// current length n, at most nsplit): the split kernel writes nothing for the others, so their records
// may hold anything, including a previous call's partials. A record with m = -inf (a chunk of padding
// only) has weight 0 and its output floats are never read: the split kernel writes only m and l there.
// The chunk weights are computed once into shared memory; each thread then sums its output element
// over the chunks with four independent chains (four record loads in flight).
constexpr int COMB_MAX_SPLITS = 1024;
template <int DH>
__global__ void __launch_bounds__(DH)
    attn_decode_combine_kernel(const float* __restrict__ work, int Hq, int nsplit, const int* __restrict__ len0p,
                               int window, int ch, __nv_bfloat16* __restrict__ out) {
    constexpr int REC = DH + 2;
    __shared__ float wgt[COMB_MAX_SPLITS];
    __shared__ float red[DH / 32];
    __shared__ float inv_l;
    pdl_trigger();  // the next kernel only prefetches weights before its own wait
    pdl_wait();
    const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x, lane = d & 31, warp = d >> 5;
    const float* wb = work + ((size_t)b * Hq + h) * nsplit * REC;
    const int n = *len0p + 1;
    const int lo = window > 0 ? max(0, n - window) : 0;
    const int used = min(nsplit, (n - 1) / ch - lo / ch + 1);
    float M = -INFINITY;
    for (int c = d; c < used; c += DH) {
        const float mi = wb[(size_t)c * REC];
        wgt[c] = mi;
        M = fmaxf(M, mi);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (lane == 0) red[warp] = M;
    __syncthreads();
    M = red[0];
#pragma unroll
    for (int w = 1; w < DH / 32; ++w) M = fmaxf(M, red[w]);
    float L = 0.f;
    for (int c = d; c < used; c += DH) {
        const float mi = wgt[c];
        const float f = mi == -INFINITY ? 0.f : exp2f(mi - M);
        wgt[c] = f;
        if (f != 0.f) L = fmaf(wb[(size_t)c * REC + 1], f, L);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    __syncthreads();
    if (lane == 0) red[warp] = L;
    __syncthreads();
    if (d == 0) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < DH / 32; ++w) t += red[w];
        inv_l = 1.f / t;
    }
    __syncthreads();
    const float* rd = wb + 2 + d;
    // a weight of 0 adds nothing; skipping it keeps unwritten output floats (NaN, inf) out of the sum
    auto term = [&](int c, float a) { return wgt[c] != 0.f ? fmaf(rd[(size_t)c * REC], wgt[c], a) : a; };
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    int c = 0;
    for (; c + 4 <= used; c += 4) {
        a0 = term(c, a0);
        a1 = term(c + 1, a1);
        a2 = term(c + 2, a2);
        a3 = term(c + 3, a3);
    }
    for (; c < used; ++c) a0 = term(c, a0);
    out[((size_t)b * Hq + h) * DH + d] = __float2bfloat16_rn(((a0 + a1) + (a2 + a3)) * inv_l);
}

// Chunks per (sequence, kv head): enough to cover every slot, or a window's keys at any alignment.
int decode_chunk(int cap, int ring) { return ring ? DEC_CHUNK_RING : (cap >= 16384 ? DEC_CHUNK : DEC_CHUNK_SHORT); }
// Per-(b, q-head, chunk) records [m, l, o[DH]].
size_t decode_records_floats(int B, int Hq, int dh, int nsplit) { return (size_t)B * Hq * nsplit * (dh + 2); }
int decode_nsplit(int cap, int window, int ring) {
    const int ch = decode_chunk(cap, ring);
    const int all = (cap + ch - 1) / ch;
    return window > 0 ? std::min(all, (window + ch - 1) / ch + 1) : all;
}
// Chunks that hold keys when the cache has n keys per sequence (slots [lo, n), chunks aligned to CH).
int decode_nsplit_for(int n, int cap, int window, int ring) {
    const int ch = decode_chunk(cap, ring);
    const int lo = window > 0 ? std::max(0, n - window) : 0;
    return std::max(1, std::min(decode_nsplit(cap, window, ring), (n - 1) / ch - lo / ch + 1));
}

template <int DH, int G, int CH>
cudaError_t decode_launch_ch(dim3 grid, const CUtensorMap& tk, const CUtensorMap& tv, const __nv_bfloat16* q, int Hq,
                             int Hkv, const int* len0, SeqMap sm, float* work, int* err, cudaStream_t st) {
    constexpr int smem = DecLayout<DH, G, CH>::SMEM;  // limit raised in attention_prepare
    return launch_pdl(attn_decode_split_kernel<DH, G, CH>, grid, dim3(DEC_THREADS), smem, st, tk, tv, q, Hq, Hkv, len0,
                      sm.meta, sm.window, sm.ring, work, err);
}

template <int DH, int G>
cudaError_t decode_launch_t(const __nv_bfloat16* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc, int B, int Hq,
                            int Hkv, int cap, const int* len0, SeqMap sm, float* work, __nv_bfloat16* out, int* err,
                            int n_keys, cudaStream_t st) {
    const int nsplit = n_keys > 0 ? decode_nsplit_for(n_keys, cap, sm.window, sm.ring) : decode_nsplit(cap, sm.window, sm.ring);
    if (nsplit > COMB_MAX_SPLITS) return cudaErrorInvalidValue;
    const dim3 grid(nsplit, Hkv, B);
    CUtensorMap tk, tv;
    if (!encode_tmap_bf16_3d(&tk, kc, DH, cap, (uint64_t)B * Hkv) || !encode_tmap_bf16_3d(&tv, vc, DH, cap, (uint64_t)B * Hkv))
        return cudaErrorInvalidValue;
    cudaError_t e;
    switch (decode_chunk(cap, sm.ring)) {
        case DEC_CHUNK_RING:
            e = decode_launch_ch<DH, G, DEC_CHUNK_RING>(grid, tk, tv, q, Hq, Hkv, len0, sm, work, err, st);
            break;
        case DEC_CHUNK_SHORT:
            e = decode_launch_ch<DH, G, DEC_CHUNK_SHORT>(grid, tk, tv, q, Hq, Hkv, len0, sm, work, err, st);
            break;
        default:
            e = decode_launch_ch<DH, G, DEC_CHUNK>(grid, tk, tv, q, Hq, Hkv, len0, sm, work, err, st);
    }
    if (e != cudaSuccess) return e;
    return launch_pdl(attn_decode_combine_kernel<DH>, dim3(Hq, B), dim3(DH), 0, st, work, Hq, nsplit, len0, sm.window,
                      decode_chunk(cap, sm.ring), out);
}

template <int DH>
cudaError_t decode_launch_dh(const __nv_bfloat16* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc, int B, int Hq,
                             int Hkv, int cap, const int* len0, SeqMap sm, float* work, __nv_bfloat16* out, int* err,
                             int n_keys, cudaStream_t st) {
    switch (Hq / Hkv) {
        case 1: return decode_launch_t<DH, 1>(q, kc, vc, B, Hq, Hkv, cap, len0, sm, work, out, err, n_keys, st);
        case 2: return decode_launch_t<DH, 2>(q, kc, vc, B, Hq, Hkv, cap, len0, sm, work, out, err, n_keys, st);
        case 4: return decode_launch_t<DH, 4>(q, kc, vc, B, Hq, Hkv, cap, len0, sm, work, out, err, n_keys, st);
        case 8: return decode_launch_t<DH, 8>(q, kc, vc, B, Hq, Hkv, cap, len0, sm, work, out, err, n_keys, st);
    }
    return cudaErrorInvalidValue;
}

// Ticket counters (one int per work item), padded to 256 bytes, at the start of the workspace.
size_t attn_tickets_floats(int B, int T, int Hq, int Hkv) {
    const size_t items = (size_t)((T + TC_BM - 1) / TC_BM) * (Hq / attn_heads_per_cta(Hq, Hkv)) * B;
    return (items + 63) / 64 * 64;
}

template <int DH, int NH>
cudaError_t prefill_launch_nh(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, int B, int T, int Hq,
                              int Hkv, const int* len0, SeqMap sm, __nv_bfloat16* out, int* err, int split,
                              int max_chunks, float* ws, cudaStream_t st) {
    using Ly = TcLayout<DH, NH>;
    const int n_qt = (T + TC_BM - 1) / TC_BM;
    dim3 grid(n_qt * max_chunks, Hq / NH, B);
    int* tickets = reinterpret_cast<int*>(ws);
    float* parts = ws ? ws + attn_tickets_floats(B, T, Hq, Hkv) : nullptr;
    return launch_pdl(attn_prefill_tc_kernel<DH, NH>, grid, dim3(Ly::THREADS), Ly::SMEM, st, tq, tk, tv, T, Hq, Hkv, len0,
                      sm.meta, sm.window, sm.ring, out, err, split, max_chunks, parts, tickets);
}

// Key range from which the persistent kernel computes its exponentials speculatively (measured: 8B
// 1x32768 5.99 -> 5.65 ms, 8B 1x8192 0.403 -> 0.389 ms, 0.6B 8x4096 0.462 -> 0.455 ms; 0.6B 1x2048,
// 21 us either way, keeps the plain order).
constexpr int kSpecMinKeys = 4096;
// Key range from which the persistent kernel alternates tiles between two softmax warpgroups (ALT).
constexpr int kAltMinKeys = 8192;

// setmaxnreg.inc waits until the registers it asks for are free, so the ALT form runs only when the
// compiled kernel was given at least the registers per thread its split hands out (checked once).
template <int DH>
bool alt_registers_cover_split() {
    static const bool ok = [] {
        cudaFuncAttributes fa{};
        if (cudaFuncGetAttributes(&fa, attn_prefill_persistent_kernel<DH, true, true>) != cudaSuccess) return false;
        const long long have = (long long)ps_threads<true>() * fa.numRegs;
        const long long need = 128LL * PS_REG_PRODUCER + 256LL * PS_REG_SOFTMAX;
        return have >= need;
    }();
    return ok;
}

template <int DH>
cudaError_t prefill_launch_dh(const __nv_bfloat16* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc, int B, int T,
                              int Hq, int Hkv, int cap, const int* len0, SeqMap sm, __nv_bfloat16* out, int* err,
                              int split, int max_chunks, float* ws, int heads, int kv_hint, cudaStream_t st) {
    CUtensorMap tq, tk, tv;
    if (!encode_tmap_bf16_3d(&tq, q, DH, T, (uint64_t)B * Hq) || !encode_tmap_bf16_3d(&tk, kc, DH, cap, (uint64_t)B * Hkv) ||
        !encode_tmap_bf16_3d(&tv, vc, DH, cap, (uint64_t)B * Hkv))
        return cudaErrorInvalidValue;
    if (split <= 0 || !ws) {
        split = 0;
        max_chunks = 1;
    }
    if (heads == 0) {
        // The persistent one-head kernel (scores two tiles ahead, score and P V MMAs from separate warps)
        // is the fastest at every measured size, the longest included (8B 1x32768: 5.93 ms against 6.60
        // for two heads per CTA); a split KV range runs in the two-heads kernel when the group allows it.
        heads = (Hq / Hkv) % 2 == 0 && split > 0 ? 2 : 1;
    }
    if (heads == 2 && (Hq / Hkv) % 2 == 0)
        return prefill_launch_nh<DH, 2>(tq, tk, tv, B, T, Hq, Hkv, len0, sm, out, err, split, max_chunks, ws, st);
    if (split > 0)
        return prefill_launch_nh<DH, 1>(tq, tk, tv, B, T, Hq, Hkv, len0, sm, out, err, split, max_chunks, ws, st);
    const long long items = (long long)((T + TC_BM - 1) / TC_BM) * Hq * B;
    const unsigned grid = (unsigned)std::min<long long>(items, device_sm_count());
    if (kv_hint >= kAltMinKeys && alt_registers_cover_split<DH>())
        return launch_pdl(attn_prefill_persistent_kernel<DH, true, true>, dim3(grid), dim3(ps_threads<true>()),
                          PsLayout<DH, true>::SMEM, st, tq, tk, tv, T, Hq, Hkv, B, len0, sm.meta, sm.window, sm.ring, out, err);
    if (kv_hint >= kSpecMinKeys)
        return launch_pdl(attn_prefill_persistent_kernel<DH, true, false>, dim3(grid), dim3(ps_threads<false>()),
                          PsLayout<DH, false>::SMEM, st, tq, tk, tv, T, Hq, Hkv, B, len0, sm.meta, sm.window, sm.ring, out, err);
    return launch_pdl(attn_prefill_persistent_kernel<DH, false, false>, dim3(grid), dim3(ps_threads<false>()),
                      PsLayout<DH, false>::SMEM, st, tq, tk, tv, T, Hq, Hkv, B, len0, sm.meta, sm.window, sm.ring, out, err);
}

}  // namespace

// Two heads of one kv group per CTA share every K/V tile load.
int attn_heads_per_cta(int Hq, int Hkv) { return (Hq / Hkv) % 2 == 0 ? 2 : 1; }

cudaError_t attn_prefill_launch(const __nv_bfloat16* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc, int B, int T,
                                int Hq, int Hkv, int dh, int cap, const int* len0, SeqMap sm, __nv_bfloat16* out,
                                int* err, int split, int max_chunks, float* ws, int heads, int kv_hint,
                                cudaStream_t st) {
    if (B <= 0 || T <= 0) return cudaSuccess;
    if (sm.ring && (sm.ring % 256 || sm.ring != cap)) return cudaErrorInvalidValue;
    if (heads < 0 || heads > 2) return cudaErrorInvalidValue;
    if (dh == 128)
        return prefill_launch_dh<128>(q, kc, vc, B, T, Hq, Hkv, cap, len0, sm, out, err, split, max_chunks, ws, heads,
                                      kv_hint, st);
    if (dh == 64)
        return prefill_launch_dh<64>(q, kc, vc, B, T, Hq, Hkv, cap, len0, sm, out, err, split, max_chunks, ws, heads,
                                     kv_hint, st);
    return cudaErrorInvalidValue;
}

size_t attn_prefill_workspace(int B, int T, int Hq, int Hkv, int dh, int max_chunks) {
    if (max_chunks <= 1) return 0;
    const int nh = attn_heads_per_cta(Hq, Hkv);
    const size_t items = (size_t)((T + TC_BM - 1) / TC_BM) * (Hq / nh) * B;
    return (attn_tickets_floats(B, T, Hq, Hkv) + items * max_chunks * nh * TC_BM * (dh + 4)) * sizeof(float);
}

void attn_prefill_split_plan(int B, int T, int Hq, int Hkv, int kv_len, int* split, int* max_chunks) {
    // Split the KV range only when the query tiles would occupy at most a quarter of the SMs over a
    // long key range (a short prefill chunk after a long context): then one CTA per query tile leaves
    // most SMs idle. On larger grids the per-CTA prologue and the merge cost more than the shorter
    // critical path saves (measured at 16 query tiles x 8 head pairs).
    const int nh = attn_heads_per_cta(Hq, Hkv);
    const long long items = (long long)((T + TC_BM - 1) / TC_BM) * (Hq / nh) * B;
    const int max_tiles = (kv_len + TC_BN - 1) / TC_BN;
    const int sms = device_sm_count();
    if (items * 4 <= sms && max_tiles >= 8) {
        const int want = (int)std::min<long long>(16, std::min<long long>(sms / items, max_tiles / 4));
        *split = (max_tiles + want - 1) / want;
        *max_chunks = (max_tiles + *split - 1) / *split;
    } else {
        *split = 0;
        *max_chunks = 1;
    }
}

size_t attn_decode_workspace(int B, int Hq, int dh, int cap, int window, int ring) {
    return decode_records_floats(B, Hq, dh, decode_nsplit(cap, window, ring)) * sizeof(float);
}

cudaError_t attn_decode_launch(const __nv_bfloat16* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc, int B, int Hq,
                               int Hkv, int dh, int cap, const int* len0, SeqMap sm, float* work, __nv_bfloat16* out,
                               int* err, int n_keys, cudaStream_t st) {
    if (B <= 0) return cudaSuccess;
    if (sm.ring && (sm.ring % DEC_CHUNK_RING || sm.ring != cap)) return cudaErrorInvalidValue;
    if (dh == 128) return decode_launch_dh<128>(q, kc, vc, B, Hq, Hkv, cap, len0, sm, work, out, err, n_keys, st);
    if (dh == 64) return decode_launch_dh<64>(q, kc, vc, B, Hq, Hkv, cap, len0, sm, work, out, err, n_keys, st);
    return cudaErrorInvalidValue;
}

int attn_decode_chunks(int n_keys, int cap, int window, int ring) {
    return n_keys > 0 ? decode_nsplit_for(n_keys, cap, window, ring) : decode_nsplit(cap, window, ring);
}

int attn_decode_kernel_count() { return 2; }

template <int DH, int G, int CH>
cudaError_t decode_prepare_one() {
    return cudaFuncSetAttribute(attn_decode_split_kernel<DH, G, CH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                DecLayout<DH, G, CH>::SMEM);
}
template <int DH, int G>
cudaError_t decode_prepare_g() {
    cudaError_t e = decode_prepare_one<DH, G, DEC_CHUNK>();
    if (e == cudaSuccess) e = decode_prepare_one<DH, G, DEC_CHUNK_SHORT>();
    if (e == cudaSuccess) e = decode_prepare_one<DH, G, DEC_CHUNK_RING>();
    return e;
}
template <int DH>
cudaError_t decode_prepare_dh() {
    cudaError_t e = decode_prepare_g<DH, 1>();
    if (e == cudaSuccess) e = decode_prepare_g<DH, 2>();
    if (e == cudaSuccess) e = decode_prepare_g<DH, 4>();
    if (e == cudaSuccess) e = decode_prepare_g<DH, 8>();
    return e;
}

cudaError_t attention_prepare() {
    const void* fns[] = {(const void*)attn_prefill_tc_kernel<128, 1>, (const void*)attn_prefill_tc_kernel<128, 2>,
                         (const void*)attn_prefill_tc_kernel<64, 1>,  (const void*)attn_prefill_tc_kernel<64, 2>,
                         (const void*)attn_prefill_persistent_kernel<128, false, false>,
                         (const void*)attn_prefill_persistent_kernel<64, false, false>,
                         (const void*)attn_prefill_persistent_kernel<128, true, false>,
                         (const void*)attn_prefill_persistent_kernel<64, true, false>,
                         (const void*)attn_prefill_persistent_kernel<128, true, true>,
                         (const void*)attn_prefill_persistent_kernel<64, true, true>};
    const int smem[] = {TcLayout<128, 1>::SMEM, TcLayout<128, 2>::SMEM, TcLayout<64, 1>::SMEM, TcLayout<64, 2>::SMEM,
                        PsLayout<128, false>::SMEM, PsLayout<64, false>::SMEM, PsLayout<128, false>::SMEM,
                        PsLayout<64, false>::SMEM, PsLayout<128, true>::SMEM,  PsLayout<64, true>::SMEM};
    for (int i = 0; i < 10; ++i) {
        cudaError_t e = cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize, smem[i]);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = decode_prepare_dh<128>();
    return e == cudaSuccess ? decode_prepare_dh<64>() : e;
}

}  // namespace q3

namespace q3 {

// Fixed scratch for the allocation-free decode entry point (qwen3_op_attention_decode_noalloc): the
// split partials of attn_decode_launch live here instead of in a caller workspace. It is part of the
// library image, so every GPU that loads the library holds it until the process exits.
constexpr size_t kDecodeNoAllocBytes = 16u << 20;
static __device__ __align__(256) float g_decode_noalloc_scratch[kDecodeNoAllocBytes / sizeof(float)];

size_t attn_decode_noalloc_max_bytes() { return kDecodeNoAllocBytes; }

// Device address of the fixed scratch on the current device. Looked up once per device, with that
// device current; host code cannot use the array's name as a device pointer.
cudaError_t attn_decode_noalloc_scratch(float** ptr) {
    static std::mutex mu;
    static float* cached[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!cached[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_noalloc_scratch);
        if (e != cudaSuccess) return e;
        cached[dev] = static_cast<float*>(p);
    }
    *ptr = cached[dev];
    return cudaSuccess;
}

}  // namespace q3
