// Tensor-core GEMM for the projections of the Qwen3 block ("A modern architecture: Qwen3",
// sections Attention, SwiGLU and The whole model: q/k/v_proj, o_proj, gate/up/down_proj and
// lm_head are bias-free nn.Linear layers, y = x W^T).
//
// C = A B^T with A [M, K] (activations) and B [N, K] (weights, nn.Linear layout), bf16 inputs,
// fp32 accumulation in tensor memory, and one of four fused epilogues:
//   EPI_BF16      C = bf16(acc)                                   (fused QKV projection)
//   EPI_SWIGLU    C = bf16(bf16(silu(bf16(g))) * bf16(u))          (gate/up; B interleaves 128-row
//                 blocks of gate and up rows, so one 256-wide tile holds matching g and u columns)
//   EPI_RESIDUAL  C = bf16(R + bf16(acc)), R may alias C            (o_proj and down_proj)
//   EPI_F32       C = acc in fp32                                   (LM head logits)
//   EPI_QKV_ROPE  fused QKV projection + per-head q_norm/k_norm + RoPE + KV-cache append: each
//                 accumulator row of a tile holds whole head vectors of one token, so the RMS over
//                 head_dim, the rotate-half pairs (i, i + dh/2) and the stores stay in one thread
//
// Design (sm_103a): a persistent kernel, one CTA per SM, 10 warps.
//   warp 0      TMA producer: 128x64 A and 256x64 B boxes (128-byte swizzle) into a 4-stage ring.
//   warp 1      TMEM owner and MMA issuer: one thread issues tcgen05.mma 128x256x16 (4 per stage)
//               into one of two 256-column fp32 accumulators, and commits stage releases and
//               accumulator-ready signals to mbarriers.
//   warps 2-9   epilogue: tcgen05.ld of the accumulator rows (warp w reads TMEM lanes 32*(w%4)..; the
//               two warps of a lane quarter take half of the columns each), fused epilogue math,
//               staged TMA stores; then release the accumulator.
// Two accumulators let tile i's epilogue overlap tile i+1's main loop. Tiles are walked M-fastest
// so concurrently running CTAs share weight (B) tiles through L2. Every mbarrier wait is bounded:
// on a timeout the kernel sets ERR_TIMEOUT, tells the other roles to stop, frees TMEM and returns.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace q3 {
namespace {

constexpr int BM = kGemmBM, BK = kGemmBK;
constexpr int A_BYTES = BM * BK * 2;
constexpr int THREADS = 192;  // skinny GEMM; the tile GEMM's count depends on its epilogue (EpiShape)
constexpr int STG_BYTES = 32768;
constexpr int EPI_LEADER = 64;  // thread 0 of warp 2 issues the epilogue's TMA loads and stores
// Epilogue warps per CTA: eight (two per TMEM lane quarter, each taking half of the columns) so the
// epilogue of a tile takes half as long. Ten warps in all cap a thread at 168 registers.
template <int EPI>
struct EpiShape {
    static constexpr int WARPS = 8;
    static constexpr int NT = 32 * WARPS;  // epilogue threads
    static constexpr int THREADS = 64 + NT;
};
// Per tile width BN (256, or 128 when 256-wide tiles cannot fill the SMs): stage size, ring depth,
// TMEM columns (two accumulators) and the instruction descriptor.
// A stage holds KSUB consecutive 64-wide K boxes of A and B: two for 128-wide tiles, so each
// barrier round trip carries as many MMA cycles as a 256-wide tile's stage.
template <int BN>
struct Cfg {
    static constexpr int KSUB = BN == 256 ? 1 : 2;
    static constexpr int B_BYTES = BN * BK * 2;  // per 64-wide K box
    static constexpr int STAGE_BYTES = KSUB * (A_BYTES + B_BYTES);
    static constexpr int STAGES = BN == 256 ? 4 : 3;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int STG_OFF = STAGES * STAGE_BYTES;  // epilogue staging: 2 boxes of [128 rows][128 B]
    static constexpr int BAR_OFF = STG_OFF + STG_BYTES;
    // 1 KB of epilogue scratch: EPI_RESIDUAL_NORM's BN gamma values, EPI_QKV_ROPE's per-row partial sums
    static constexpr int GAMMA_OFF = BAR_OFF + 256;
    static constexpr int SMEM_BYTES = GAMMA_OFF + 1024 + 1024;
    static constexpr uint32_t IDESC = idesc_bf16(BM, BN);
};

struct Tile {
    int m0, n0;
};
// Tiles are walked in groups of up to 32 M-tiles: within a group M runs fastest, so the CTAs resident
// at one time share a few weight (B) tiles and a bounded slice of A through L2.
constexpr int GROUP_M = 32;
template <int BN>
__device__ __forceinline__ Tile tile_of(int t, int m_tiles, int n_tiles) {
    const int per_group = GROUP_M * n_tiles;
    const int g = t / per_group, first = g * GROUP_M;
    const int gm = min(GROUP_M, m_tiles - first);
    const int local = t - g * per_group;
    return {(first + local % gm) * BM, (local / gm) * BN};
}

// Fused epilogue of the QKV projection for one accumulator row (token) of a 256-wide tile: the
// projection output is rounded to bf16 as the unfused path stores it, then V heads go to the cache
// unchanged and Q/K heads get RMSNorm over head_dim (fp32 reduce, bf16 cast, then gamma) and RoPE
// (bf16(bf16(a c) + bf16(-b s)), bf16(bf16(b c) + bf16(a s)) for the pair (i, i + dh/2)).
// Address of 16-byte chunk u (0..15) of tile row r in the staging buffer: two TMA boxes of
// [128 rows][128 bytes] in the 128-byte swizzle pattern (chunk index XOR row % 8).
__device__ __forceinline__ uint8_t* stg_chunk(uint8_t* stg, int r, int u) {
    return stg + (u >> 3) * 16384 + r * 128 + (((u & 7) ^ (r & 7)) << 4);
}

struct EpiSync {
    uint64_t* res_bar;  // residual tile arrival (TMA load, tx count)
    uint32_t res_phase;
    volatile int* fail;  // set by any epilogue warp whose wait gave up
};

// Make a warp's wait outcome uniform over the NT epilogue threads: every thread reaches the barrier
// (the waits before it are bounded), so all epilogue warps take the same branch afterwards.
template <int NT>
__device__ __forceinline__ bool epi_agree(bool ok, volatile int* fail) {
    if (!__all_sync(0xffffffffu, ok) && (threadIdx.x & 31) == 0) *fail = 1;
    named_barrier(1, NT);
    return *fail == 0;
}

// Staging-buffer hand-off between passes: the previous TMA store must have read it.
template <int NT>
__device__ __forceinline__ void stg_acquire() {
    if (threadIdx.x == EPI_LEADER) bulk_wait_read();
    named_barrier(1, NT);
}
// Publish the staging buffer (generic-proxy writes) to the TMA store and issue it.
template <int NT>
__device__ __forceinline__ void stg_store(uint8_t* stg, const CUtensorMap* tmC, int x0, int x1, int y) {
    fence_proxy_async_smem();
    named_barrier(1, NT);
    if (threadIdx.x == EPI_LEADER) {
        tma_store_2d(tmC, stg, x0, y);
        tma_store_2d(tmC, stg + 16384, x1, y);
        bulk_commit();
    }
}

// Load 128 consecutive accumulator columns of this thread's row (4 loads, one wait).
__device__ __forceinline__ void tmem_ld_128(uint32_t taddr, uint32_t (&r)[128]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(taddr + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&r[c * 32]));
    tmem_ld_wait();
}

// Epilogue of one tile for the staged epilogues (BF16, RESIDUAL, SWIGLU, F32), eight warps: warp half
// `hf` (0 or 1) of each TMEM lane quarter takes the second 64-column box (bf16; 32 columns fp32) of
// every 128-column pass. The accumulator is released (acc_empty) as soon as a thread's last columns
// are in registers; outputs go through the staging buffer and TMA stores, so each warp writes whole
// swizzled rows of its box to shared memory and the copy to global memory is one coalesced bulk
// operation per box. Returns false if a wait gave up.
template <int EPI, int BN>
__device__ __forceinline__ bool epilogue_staged(const GemmArgs& a, const CUtensorMap* tmC, const CUtensorMap* tmR,
                                                uint8_t* stg, EpiSync& es, uint32_t tacc, int r, int hf, int m0,
                                                int n0, uint64_t* acc_empty, uint64_t* acc_full, uint32_t aph,
                                                volatile int* abort_flag) {
    constexpr int NT = EpiShape<EPI>::NT;
    // passes of 128 bf16 (or 64 fp32) output columns, each filling the 32 KB staging buffer
    constexpr int PASSES = EPI == EPI_SWIGLU ? 1 : (EPI == EPI_F32 ? BN / 64 : BN / 128);
#pragma unroll 1
    for (int p = 0; p < PASSES; ++p) {
        stg_acquire<NT>();
        if constexpr (EPI == EPI_RESIDUAL) {
            if (threadIdx.x == EPI_LEADER) {
                mbar_expect_tx(es.res_bar, STG_BYTES);
                tma_load_2d(stg, tmR, es.res_bar, n0 + p * 128, m0);
                tma_load_2d(stg + 16384, tmR, es.res_bar, n0 + p * 128 + 64, m0);
            }
        }
        if (p == 0) {
            // the accumulator of this tile
            const bool w = mbar_wait_suspend(acc_full, aph, abort_flag);
            if (!epi_agree<NT>(w, es.fail)) return false;
            tc_fence_after();
        }
        if constexpr (EPI == EPI_SWIGLU) {
            // gate columns [0, BN/2), up columns [BN/2, BN): this half's 64 outputs are gate columns
            // [64 hf, 64 hf + 64) times the matching up columns (BN = 256)
#pragma unroll 1
            for (int sub = 0; sub < 2; ++sub) {  // 32 outputs at a time (registers of a 10-warp CTA)
                uint32_t g[32], u[32];
                tmem_ld_32x32b_x32(tacc + hf * 64 + sub * 32, g);
                tmem_ld_32x32b_x32(tacc + BN / 2 + hf * 64 + sub * 32, u);
                tmem_ld_wait();
                if (sub == 1) {
                    tc_fence_before();
                    mbar_arrive(acc_empty);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t wv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        // columns j, j + 1 in paired fp32: silu(g) = g / (1 + 2^(-g log2 e))
                        const int j = q * 8 + 2 * e;
                        const uint32_t gb = pack_bf16(__uint_as_float(g[j]), __uint_as_float(g[j + 1]));
                        const float2 gf = make_float2(bf16_lo(gb), bf16_hi(gb));
                        const float2 t = mul2(gf, make_float2(-kLog2e, -kLog2e));
                        const float2 den = add2(make_float2(ex2_approx(t.x), ex2_approx(t.y)), make_float2(1.f, 1.f));
                        const float2 sv = mul2(gf, make_float2(rcp_approx(den.x), rcp_approx(den.y)));
                        const uint32_t sb = pack_bf16(sv.x, sv.y);
                        const uint32_t ub = pack_bf16(__uint_as_float(u[j]), __uint_as_float(u[j + 1]));
                        const float2 pv = mul2(make_float2(bf16_lo(sb), bf16_hi(sb)), make_float2(bf16_lo(ub), bf16_hi(ub)));
                        wv[e] = pack_bf16(pv.x, pv.y);
                    }
                    *reinterpret_cast<uint4*>(stg_chunk(stg, r, hf * 8 + sub * 4 + q)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
            }
            stg_store<NT>(stg, tmC, n0 / 2, n0 / 2 + 64, m0);
        } else if constexpr (EPI == EPI_F32) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tacc + p * 64 + hf * 32, v);
            tmem_ld_wait();
            if (p == PASSES - 1) {
                tc_fence_before();
                mbar_arrive(acc_empty);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                *reinterpret_cast<uint4*>(stg_chunk(stg, r, hf * 8 + u)) =
                    make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
            stg_store<NT>(stg, tmC, n0 + p * 64, n0 + p * 64 + 32, m0);
        } else {
            uint32_t v[64];
            tmem_ld_32x32b_x32(tacc + p * 128 + hf * 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            tmem_ld_32x32b_x32(tacc + p * 128 + hf * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            tmem_ld_wait();
            if (p == PASSES - 1) {
                tc_fence_before();
                mbar_arrive(acc_empty);
            }
            if constexpr (EPI == EPI_RESIDUAL) {
                const bool w = mbar_wait_suspend(es.res_bar, es.res_phase & 1, abort_flag);
                ++es.res_phase;
                if (!epi_agree<NT>(w, es.fail)) return false;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                uint4* cp = reinterpret_cast<uint4*>(stg_chunk(stg, r, hf * 8 + u));
                uint32_t wv[4];
                if constexpr (EPI == EPI_RESIDUAL) {
                    const uint4 q = *cp;
                    const uint32_t rr[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        wv[e] = pack_bf16(bf16_lo(rr[e]) + rbf(__uint_as_float(v[8 * u + 2 * e])),
                                          bf16_hi(rr[e]) + rbf(__uint_as_float(v[8 * u + 2 * e + 1])));
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        wv[e] = pack_bf16(__uint_as_float(v[8 * u + 2 * e]), __uint_as_float(v[8 * u + 2 * e + 1]));
                }
                *cp = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
            stg_store<NT>(stg, tmC, n0 + p * 128, n0 + p * 128 + 64, m0);
        }
    }
    return true;
}

// Residual epilogue followed by the next RMSNorm ("A modern architecture: Qwen3", section RMSNorm and
// the pre-norm block) for one of the csize column tiles of a row block, which run concurrently on
// different CTAs: X = bf16(R + bf16(acc)) is stored as in EPI_RESIDUAL and kept in tensor memory
// (packed over the accumulator's own columns); each row's sum of squares over the tile goes to
// part[row block][rank][row]. When all csize CTAs have arrived on the row block's counter, the
// partial sums are added in rank order (the same in every CTA), r = rsqrt(sum / N + eps), and
// Y = bf16(gamma * bf16(X * r)) is stored through the v map. The accumulator is released last.
template <int BN>
__device__ __forceinline__ bool epilogue_residual_norm(const GemmArgs& a, const CUtensorMap* tmC, const CUtensorMap* tmR,
                                                       const CUtensorMap* tmY, uint8_t* stg, EpiSync& es, uint32_t tacc,
                                                       int r, int hf, int m0, int n0, int rank, int csize,
                                                       const uint8_t* gam, uint64_t* acc_empty, uint64_t* acc_full,
                                                       uint32_t aph, volatile int* abort_flag) {
    constexpr int NT = EpiShape<EPI_RESIDUAL_NORM>::NT;
    constexpr int PASSES = BN / 128;
    float ss = 0.f;
#pragma unroll 1
    for (int p = 0; p < PASSES; ++p) {
        stg_acquire<NT>();
        if (threadIdx.x == EPI_LEADER) {
            mbar_expect_tx(es.res_bar, STG_BYTES);
            tma_load_2d(stg, tmR, es.res_bar, n0 + p * 128, m0);
            tma_load_2d(stg + 16384, tmR, es.res_bar, n0 + p * 128 + 64, m0);
        }
        if (p == 0) {
            const bool w = mbar_wait_suspend(acc_full, aph, abort_flag);
            if (!epi_agree<NT>(w, es.fail)) return false;
            tc_fence_after();
        }
        // this half's 64 columns of the pass (staging box hf)
        const uint32_t ta = tacc + p * 128 + hf * 64;
        uint32_t v[64];
        tmem_ld_32x32b_x32(ta, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld_32x32b_x32(ta + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        tmem_ld_wait();
        {
            const bool w = mbar_wait_suspend(es.res_bar, es.res_phase & 1, abort_flag);
            ++es.res_phase;
            if (!epi_agree<NT>(w, es.fail)) return false;
        }
        uint32_t xw[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            uint4* cp = reinterpret_cast<uint4*>(stg_chunk(stg, r, hf * 8 + u));
            const uint4 q = *cp;
            const uint32_t rr[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t xv = pack_bf16(bf16_lo(rr[e]) + rbf(__uint_as_float(v[8 * u + 2 * e])),
                                              bf16_hi(rr[e]) + rbf(__uint_as_float(v[8 * u + 2 * e + 1])));
                xw[4 * u + e] = xv;
                ss = fmaf(bf16_lo(xv), bf16_lo(xv), ss);
                ss = fmaf(bf16_hi(xv), bf16_hi(xv), ss);
            }
            *cp = make_uint4(xw[4 * u], xw[4 * u + 1], xw[4 * u + 2], xw[4 * u + 3]);
        }
        // X packed over the first 32 of the columns this thread has just read
        tmem_st_32x32b_x32(ta, xw);
        stg_store<NT>(stg, tmC, n0 + p * 128, n0 + p * 128 + 64, m0);
    }
    tmem_st_wait();
    // this half-tile's partial sums of squares, then meet the row block's other column tiles (the
    // releasing increment publishes every epilogue thread's sum, ordered before it by the barrier)
    const size_t rb = (size_t)(m0 / BM);
    unsigned* arrive = a.norm.count + 2 * rb;
    a.norm.part[((rb * csize + rank) * 2 + hf) * BM + r] = ss;
    named_barrier(1, NT);
    bool met = true;
    if (threadIdx.x == EPI_LEADER) {
        red_add_release_gpu(arrive, 1u);
        const uint64_t t0 = globaltimer();
        for (uint32_t i = 1; ld_acquire_gpu(arrive) < (unsigned)csize; ++i) {
            if ((i & 63u) == 0 && (*abort_flag || globaltimer() - t0 > kWaitTimeoutNs)) {
                met = false;
                break;
            }
        }
    }
    if (!epi_agree<NT>(met, es.fail)) return false;
    // the row block's partial sums (at most 8 column tiles x 2 halves), all loads in flight at once, then
    // added in a fixed order: column tile, then half
    float pv[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) pv[q] = q < 2 * csize ? __ldcg(a.norm.part + (rb * csize * 2 + q) * BM + r) : 0.f;
    float tot = 0.f;
#pragma unroll
    for (int q = 0; q < 16; ++q)
        if (q < 2 * csize) tot += pv[q];
    const float rn = __frsqrt_rn(tot / (float)(csize * BN) + a.norm.eps);
#pragma unroll 1
    for (int p = 0; p < PASSES; ++p) {
        uint32_t xw[32];
        tmem_ld_32x32b_x32(tacc + p * 128 + hf * 64, xw);
        tmem_ld_wait();
        stg_acquire<NT>();
        const uint4* gp = reinterpret_cast<const uint4*>(gam + (p * 128 + hf * 64) * 2);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const uint4 gv = gp[u];
            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t xv = xw[4 * u + e];
                o[e] = pack_bf16(bf16_lo(gw[e]) * rbf(bf16_lo(xv) * rn), bf16_hi(gw[e]) * rbf(bf16_hi(xv) * rn));
            }
            *reinterpret_cast<uint4*>(stg_chunk(stg, r, hf * 8 + u)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        stg_store<NT>(stg, tmY, n0 + p * 128, n0 + p * 128 + 64, m0);
    }
    tc_fence_before();
    mbar_arrive(acc_empty);
    // the last CTA of the row block to get here resets its counters for the next launch (every CTA
    // has passed the meeting once it has counted itself out)
    if (threadIdx.x == EPI_LEADER && atomicAdd(arrive + 1, 1u) == (unsigned)csize - 1) {
        arrive[0] = 0;
        arrive[1] = 0;
    }
    return true;
}

// Fused QKV epilogue for one tile: per head of the tile, each thread (one token row) rounds its
// projection to bf16, then V heads are copied and Q/K heads get RMSNorm over head_dim (fp32 reduce,
// bf16 cast, then gamma) and RoPE (bf16(bf16(a c) + bf16(-b s)), bf16(bf16(b c) + bf16(a s)) for the
// pair (i, i + dh/2)). The two warp halves of a TMEM lane quarter split each head's rotation pairs:
// half hf takes i in [hf dh/4, (hf + 1) dh/4) and the partners i + dh/2, and the halves add their
// partial sums of squares through shared memory (64-thread barriers per lane quarter). When the
// tile's 128 rows are consecutive tokens of one sequence (prefill with T % 128 == 0), each head's
// [128 x dh] block is written through the staging buffer with one 3-D TMA store into Q [B*Hq][T][dh] or
// the cache [B*Hkv][cap][dh]; otherwise (decode) rows are stored directly.
template <int DH, int BN>
__device__ __forceinline__ bool epilogue_qkv_rope(const GemmArgs& a, const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                                  const CUtensorMap* tmV, uint8_t* stg, EpiSync& es, uint32_t tacc,
                                                  int r, int hf, int m0, int n0, uint64_t* acc_empty,
                                                  uint64_t* acc_full, uint32_t aph, volatile int* xss_raw,
                                                  volatile int* abort_flag) {
    constexpr int NT = EpiShape<EPI_QKV_ROPE>::NT;
    volatile float(*xss)[128] = reinterpret_cast<volatile float(*)[128]>(xss_raw);  // [half][row] partial sums
    const QkvRopeArgs& q = a.qkv;
    const int row = m0 + r;
    const bool row_ok = row < a.M;
    const int len0 = *q.len0;
    // whole 128-row blocks go out by TMA, unless a rolling buffer could wrap inside the block
    const bool staged = (q.T % BM) == 0 && (!q.rolling || len0 % BM == 0);
    const int b = row_ok ? row / q.T : 0, t = row_ok ? row % q.T : 0;
    constexpr int HALF = DH / 2, QC = DH / 4;  // QC: columns per side of this half
    constexpr int NHEAD = BN / DH;
    {
        const bool w = mbar_wait_suspend(acc_full, aph, abort_flag);
        if (staged) {
            if (!epi_agree<NT>(w, es.fail)) return false;
        } else if (!__all_sync(0xffffffffu, w)) {
            return false;
        }
        tc_fence_after();
    }
    const int slot = len0 + t;
    const int pos = q.meta ? slot_position(slot, q.meta[0], q.meta[kSeqMetaHead + b]) : slot;
    const int phys = q.rolling ? slot % q.cap : slot;
    const int pair_bar = 2 + (r >> 5);  // the two warps of this lane quarter
#pragma unroll 1
    for (int lh = 0; lh < NHEAD; ++lh) {
        const int hg = n0 / DH + lh;
        uint32_t x1[QC], x2[QC];  // columns [hf QC, hf QC + QC) and [HALF + hf QC, ...) of the head
        const uint32_t c1 = tacc + lh * DH + hf * QC, c2 = c1 + HALF;
        if constexpr (QC == 32) {
            tmem_ld_32x32b_x32(c1, *reinterpret_cast<uint32_t(*)[32]>(&x1[0]));
            tmem_ld_32x32b_x32(c2, *reinterpret_cast<uint32_t(*)[32]>(&x2[0]));
        } else {
            tmem_ld_32x32b_x16(c1, x1);
            tmem_ld_32x32b_x16(c2, x2);
        }
        tmem_ld_wait();
        if (lh == NHEAD - 1) {
            tc_fence_before();
            mbar_arrive(acc_empty);
        }
        const int kind = hg < q.Hq ? 0 : (hg < q.Hq + q.Hkv ? 1 : 2);  // q, k, v
        uint32_t o1[QC / 2], o2[QC / 2];  // packed bf16 outputs of the two sides
        if (kind == 2) {
#pragma unroll
            for (int j = 0; j < QC / 2; ++j) {
                o1[j] = pack_bf16(__uint_as_float(x1[2 * j]), __uint_as_float(x1[2 * j + 1]));
                o2[j] = pack_bf16(__uint_as_float(x2[2 * j]), __uint_as_float(x2[2 * j + 1]));
            }
        } else {
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < QC; ++j) {
                const float xa = rbf(__uint_as_float(x1[j])), xb = rbf(__uint_as_float(x2[j]));
                x1[j] = __float_as_uint(xa);
                x2[j] = __float_as_uint(xb);
                ss = fmaf(xa, xa, ss);
                ss = fmaf(xb, xb, ss);
            }
            xss[hf][r] = ss;
            named_barrier(pair_bar, 64);
            const float tot = xss[0][r] + xss[1][r];  // same order in both halves
            named_barrier(pair_bar, 64);             // both have read before the next head's write
            const float rn = __frsqrt_rn(tot / (float)DH + q.eps);
            const __nv_bfloat16* gam = kind == 0 ? q.q_gamma : q.k_gamma;
            const __nv_bfloat16* cs = q.table + (size_t)(row_ok ? pos : 0) * DH;
            // bf16x2 arithmetic: each packed multiply / add rounds once to bf16, as the definition does
#pragma unroll
            for (int vv = 0; vv < QC / 8; ++vv) {
                const int v = hf * (QC / 8) + vv;  // 8-element group of the first half of the head
                const uint4 g0 = __ldg(reinterpret_cast<const uint4*>(gam) + v);
                const uint4 g1 = __ldg(reinterpret_cast<const uint4*>(gam + HALF) + v);
                const uint4 cc = __ldg(reinterpret_cast<const uint4*>(cs) + v);
                const uint4 sn = __ldg(reinterpret_cast<const uint4*>(cs + HALF) + v);
                const uint32_t G0[4] = {g0.x, g0.y, g0.z, g0.w}, G1[4] = {g1.x, g1.y, g1.z, g1.w};
                const uint32_t C[4] = {cc.x, cc.y, cc.z, cc.w}, S[4] = {sn.x, sn.y, sn.z, sn.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = 8 * vv + 2 * e;
                    // normalised, cast, then times gamma: a = first-half pair, bb = second-half pair
                    const uint32_t na = pack_bf16(__uint_as_float(x1[j]) * rn, __uint_as_float(x1[j + 1]) * rn);
                    const uint32_t nb = pack_bf16(__uint_as_float(x2[j]) * rn, __uint_as_float(x2[j + 1]) * rn);
                    const __nv_bfloat162 av = __hmul2_rn(as_bf2(G0[e]), as_bf2(na));
                    const __nv_bfloat162 bv = __hmul2_rn(as_bf2(G1[e]), as_bf2(nb));
                    const __nv_bfloat162 co = as_bf2(C[e]), si = as_bf2(S[e]);
                    o1[4 * vv + e] = as_u32(__hsub2(__hmul2_rn(av, co), __hmul2_rn(bv, si)));
                    o2[4 * vv + e] = as_u32(__hadd2(__hmul2_rn(bv, co), __hmul2_rn(av, si)));
                }
            }
        }
        // 16-byte chunks of the head row: this half's first-side chunks are hf QC/8 .. and its
        // second-side chunks HALF/8 + hf QC/8 ..
        const int u1 = hf * (QC / 8), u2 = HALF / 8 + hf * (QC / 8);
        if (staged) {
            stg_acquire<NT>();
#pragma unroll
            for (int vv = 0; vv < QC / 8; ++vv) {
                *reinterpret_cast<uint4*>(stg_chunk(stg, r, u1 + vv)) =
                    make_uint4(o1[4 * vv], o1[4 * vv + 1], o1[4 * vv + 2], o1[4 * vv + 3]);
                *reinterpret_cast<uint4*>(stg_chunk(stg, r, u2 + vv)) =
                    make_uint4(o2[4 * vv], o2[4 * vv + 1], o2[4 * vv + 2], o2[4 * vv + 3]);
            }
            fence_proxy_async_smem();
            named_barrier(1, NT);
            if (threadIdx.x == EPI_LEADER) {
                const int bt = m0 / q.T, t0 = m0 % q.T;
                const CUtensorMap* map = kind == 0 ? tmQ : (kind == 1 ? tmK : tmV);
                const int y = kind == 0 ? t0 : (q.rolling ? (len0 + t0) % q.cap : len0 + t0);
                const int z = kind == 0 ? bt * q.Hq + hg : bt * q.Hkv + (kind == 1 ? hg - q.Hq : hg - q.Hq - q.Hkv);
#pragma unroll
                for (int c = 0; c < DH / 64; ++c) tma_store_3d(map, stg + c * 16384, c * 64, y, z);
                bulk_commit();
            }
        } else if (row_ok) {
            __nv_bfloat16* dst = kind == 0 ? q.q_out + (((size_t)b * q.Hq + hg) * q.T + t) * DH
                               : kind == 1 ? q.k_cache + (((size_t)b * q.Hkv + (hg - q.Hq)) * q.cap + phys) * DH
                                           : q.v_cache + (((size_t)b * q.Hkv + (hg - q.Hq - q.Hkv)) * q.cap + phys) * DH;
#pragma unroll
            for (int vv = 0; vv < QC / 8; ++vv) {
                reinterpret_cast<uint4*>(dst)[u1 + vv] = make_uint4(o1[4 * vv], o1[4 * vv + 1], o1[4 * vv + 2], o1[4 * vv + 3]);
                reinterpret_cast<uint4*>(dst)[u2 + vv] = make_uint4(o2[4 * vv], o2[4 * vv + 1], o2[4 * vv + 2], o2[4 * vv + 3]);
            }
        }
    }
    return true;
}

// Every mbarrier wait in the GEMM kernels parks the waiting threads with a suspend-time hint instead of
// polling: the epilogue warps wait out each tile's MMAs and the producers wait for ring stages, and their
// polling took issue slots and power from a step that runs at the power cap (measured: 0.6B 1x2048 prefill
// 750k -> 760k tokens/s, 8B decode 14.49 -> 14.42 ms, the 8B 1x32768 prefill unchanged).
template <int EPI, int BN>
__global__ void __launch_bounds__(EpiShape<EPI>::THREADS, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmR,
                        const __grid_constant__ CUtensorMap tmV, const GemmArgs args) {
    using C = Cfg<BN>;
    constexpr int STAGES = C::STAGES, STAGE_BYTES = C::STAGE_BYTES, TMEM_COLS = C::TMEM_COLS;
    constexpr uint32_t IDESC = C::IDESC;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t* stg = smem + C::STG_OFF;
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* empty_bar = full_bar + STAGES;
    uint64_t* acc_full = empty_bar + STAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* res_bar = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(res_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* epi_fail = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tiles = (args.M + BM - 1) / BM, n_tiles = (args.N + BN - 1) / BN;
    constexpr int KSUB = C::KSUB;
    const int k_blocks = (args.K + BK * KSUB - 1) / (BK * KSUB);  // stages per tile
    // Work walk: tiles blockIdx.x, + gridDim.x, ... With the fused norm the tiles go row block by row
    // block and the grid is a multiple of n_tiles, so the column tiles of a row block run at the same
    // time on consecutive CTAs and a CTA keeps one column tile (rank).
    constexpr bool RN = EPI == EPI_RESIDUAL_NORM;
    const int rank = RN ? (int)blockIdx.x % n_tiles : 0;
    const int first = (int)blockIdx.x, step = (int)gridDim.x, limit = m_tiles * n_tiles;
    auto tile_at = [&](int t) -> Tile {
        return RN ? Tile{t / n_tiles * BM, t % n_tiles * BN} : tile_of<BN>(t, m_tiles, n_tiles);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], EpiShape<EPI>::NT);
        }
        mbar_init(res_bar, 1);
        *abort_flag = 0;
        *epi_fail = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if constexpr (EPI != EPI_QKV_ROPE) tma_prefetch_desc(&tmC);
        if constexpr (EPI == EPI_RESIDUAL || RN) tma_prefetch_desc(&tmR);
        if constexpr (RN) tma_prefetch_desc(&tmV);
        if constexpr (EPI == EPI_QKV_ROPE) {
            if (args.qkv.T % BM == 0) {
                tma_prefetch_desc(&tmC);
                tma_prefetch_desc(&tmR);
                tma_prefetch_desc(&tmV);
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    bool ok = true;
    // B boxes of the first tile's first stages, issued before the wait on the previous kernel when
    // the weights do not depend on it (their DRAM latency then overlaps that kernel's tail)
    auto load_b = [&](uint8_t* sa, uint64_t* bar, int kb, int n0) {
#pragma unroll
        for (int j = 0; j < KSUB; ++j)
#pragma unroll
            for (int nb = 0; nb < BN / kGemmBoxN; ++nb)
                tma_load_2d(sa + KSUB * A_BYTES + j * C::B_BYTES + nb * kGemmBoxN * BK * 2, &tmB, bar,
                            (kb * KSUB + j) * BK, n0 + nb * kGemmBoxN);
    };
    int pre = 0;
    if (warp == 0 && lane == 0 && args.b_independent && first < limit) {
        const Tile tl = tile_at(first);
        pre = min(STAGES, k_blocks);
        for (int kb = 0; kb < pre; ++kb) {
            mbar_expect_tx(&full_bar[kb], STAGE_BYTES);
            load_b(smem + kb * STAGE_BYTES, &full_bar[kb], kb, tl.n0);
        }
    }
    pdl_wait();  // inputs of this GEMM come from the previous kernel
    pdl_trigger();

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer
        int it = 0;
        for (int t = first; t < limit && ok; t += step) {
            const Tile tl = tile_at(t);
            for (int kb = 0; kb < k_blocks; ++kb, ++it) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1;
                uint8_t* sa = smem + s * STAGE_BYTES;
                if (it >= pre) {
                    if (!mbar_wait_suspend(&empty_bar[s], ph ^ 1, abort_flag)) { ok = false; break; }
                    mbar_expect_tx(&full_bar[s], STAGE_BYTES);
                    load_b(sa, &full_bar[s], kb, tl.n0);
                }
#pragma unroll
                for (int j = 0; j < KSUB; ++j)  // boxes past K read as zeros
                    tma_load_2d(sa + j * A_BYTES, &tmA, &full_bar[s], (kb * KSUB + j) * BK, tl.m0);
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        int it = 0, local = 0;
        for (int t = first; t < limit && ok; t += step, ++local) {
            const int acc = local & 1;
            const uint32_t aph = (local >> 1) & 1;
            if (!mbar_wait_suspend(&acc_empty[acc], aph ^ 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * BN;
            for (int kb = 0; kb < k_blocks; ++kb, ++it) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1;
                if (!mbar_wait_suspend(&full_bar[s], ph, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sa = smem_u32(smem + s * STAGE_BYTES);
#pragma unroll
                for (int j = 0; j < KSUB; ++j) {
                    const uint64_t adesc = sdesc_kmajor_sw128(sa + j * A_BYTES);
                    const uint64_t bdesc = sdesc_kmajor_sw128(sa + KSUB * A_BYTES + j * C::B_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        umma_bf16_ss(d_tmem, adesc + 2 * k, bdesc + 2 * k, IDESC, (kb | j | k) != 0);
                }
                umma_commit(&empty_bar[s]);
            }
            if (!ok) break;
            umma_commit(&acc_full[acc]);
        }
    } else if (warp >= 2) {
        // ---------------- epilogue
        const int quarter = warp & 3, hf = (warp - 2) >> 2;  // hf: which half of the columns (8 warps)
        const int r = quarter * 32 + lane;                     // tile row = TMEM lane
        EpiSync es{res_bar, 0, epi_fail};
        if constexpr (RN) {  // this CTA's column tile is fixed: stage its gamma values once
            const int et = threadIdx.x - 64;
            if (et < BN / 8)
                reinterpret_cast<uint4*>(smem + C::GAMMA_OFF)[et] =
                    __ldg(reinterpret_cast<const uint4*>(args.norm.gamma + rank * BN) + et);
            named_barrier(1, EpiShape<EPI>::NT);
        }
        int local = 0;
        for (int t = first; t < limit; t += step, ++local) {
            const int acc = local & 1;
            const uint32_t aph = (local >> 1) & 1;
            const Tile tl = tile_at(t);
            const uint32_t tacc = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
            if constexpr (EPI == EPI_QKV_ROPE) {
                volatile int* xss = reinterpret_cast<volatile int*>(smem + C::GAMMA_OFF);
                const bool w = args.qkv.dh == 128
                                   ? epilogue_qkv_rope<128, BN>(args, &tmC, &tmR, &tmV, stg, es, tacc, r, hf, tl.m0,
                                                                tl.n0, &acc_empty[acc], &acc_full[acc], aph, xss,
                                                                abort_flag)
                                   : epilogue_qkv_rope<64, BN>(args, &tmC, &tmR, &tmV, stg, es, tacc, r, hf, tl.m0,
                                                               tl.n0, &acc_empty[acc], &acc_full[acc], aph, xss,
                                                               abort_flag);
                if (!w) {
                    ok = false;
                    break;
                }
            } else if constexpr (RN) {
                if (!epilogue_residual_norm<BN>(args, &tmC, &tmR, &tmV, stg, es, tacc, r, hf, tl.m0, tl.n0, rank,
                                                n_tiles, smem + C::GAMMA_OFF, &acc_empty[acc], &acc_full[acc], aph,
                                                abort_flag)) {
                    ok = false;
                    break;
                }
            } else {
                if (!epilogue_staged<EPI, BN>(args, &tmC, &tmR, stg, es, tacc, r, hf, tl.m0, tl.n0, &acc_empty[acc],
                                              &acc_full[acc], aph, abort_flag)) {
                    ok = false;
                    break;
                }
            }
        }
        // shared memory must outlive the reads of the last TMA stores; their global writes complete
        // with the grid, which the next kernel's dependency wait (or stream order) covers
        if (threadIdx.x == EPI_LEADER) bulk_wait_read();
    }
    if (!ok) {
        *abort_flag = 1;
        if (args.err) atomicOr(args.err, ERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}


// ------------------------------------------------------------------------------ skinny (decode)
// Weight-streaming GEMM for decode batches, persistent: a work item is 128 weight rows x one K chunk
// (split), and each CTA walks items c, c + G, ... . Warp 0 streams 128x64 weight boxes and 64x64
// activation boxes through an 8-stage ring without draining it between items, warp 1 issues
// tcgen05.mma M=128 (weight rows) x N=MP (activation rows) x K=16 into one of two MP-column TMEM
// accumulators, and warps 2-5 read a finished accumulator (thread = weight row) and store it into the
// item's fp32 slice of the workspace (or straight to the output when K is not split) while the next
// item accumulates. With few rows the kernel is bound by reading the weights once.
constexpr int SK_STAGES = 8;
constexpr int SK_W_BYTES = 128 * BK * 2;
constexpr int SK_X_BYTES = kSkinnyRowsBox * BK * 2;
constexpr int SK_STAGE_BYTES = SK_W_BYTES + SK_X_BYTES;
constexpr int SK_SMEM = SK_STAGES * SK_STAGE_BYTES + 256 + 1024;

template <int MP>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       const SkinnyArgs args) {
    constexpr uint32_t IDESC = idesc_bf16(128, MP);
    constexpr uint32_t TCOLS = MP < 32 ? 32 : MP;  // columns of one accumulator; two are allocated
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + SK_STAGES * SK_STAGE_BYTES);
    uint64_t* empty_bar = full_bar + SK_STAGES;
    uint64_t* acc_full = empty_bar + SK_STAGES;  // [2]
    uint64_t* acc_empty = acc_full + 2;          // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row_blocks = (args.N + 127) / 128;
    const int items = row_blocks * args.splits;
    const int k_blocks = (args.K + BK - 1) / BK;
    const int per = (k_blocks + args.splits - 1) / args.splits;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SK_STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 128);
        }
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 2 * TCOLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    // K range [kb0, kb1) of an item (item = split * row_blocks + row block)
    auto k_range = [&](int item, int& kb0, int& kb1) {
        kb0 = (item / row_blocks) * per;
        kb1 = min(k_blocks, kb0 + per);
    };
    // weight boxes of the first item's first stages, issued before the wait on the previous kernel
    // when the weights do not depend on it
    int pre = 0;
    if (warp == 0 && lane == 0 && args.w_independent && (int)blockIdx.x < items) {
        int kb0, kb1;
        k_range(blockIdx.x, kb0, kb1);
        const int n0 = (blockIdx.x % row_blocks) * 128;
        pre = max(0, min(SK_STAGES, kb1 - kb0));
        for (int i = 0; i < pre; ++i) {
            mbar_expect_tx(&full_bar[i], SK_STAGE_BYTES);
            tma_load_2d(smem + i * SK_STAGE_BYTES, &tmW, &full_bar[i], (kb0 + i) * BK, n0);
        }
    }
    pdl_wait();
    pdl_trigger();

    if (warp == 0 && lane == 0) {
        int it = 0;
        for (int item = blockIdx.x; item < items && ok; item += gridDim.x) {
            int kb0, kb1;
            k_range(item, kb0, kb1);
            const int n0 = (item % row_blocks) * 128;
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int s = it % SK_STAGES;
                uint8_t* st = smem + s * SK_STAGE_BYTES;
                if (it >= pre) {
                    if (!mbar_wait_suspend(&empty_bar[s], ((it / SK_STAGES) & 1) ^ 1, abort_flag)) { ok = false; break; }
                    mbar_expect_tx(&full_bar[s], SK_STAGE_BYTES);
                    tma_load_2d(st, &tmW, &full_bar[s], kb * BK, n0);
                }
                tma_load_2d(st + SK_W_BYTES, &tmX, &full_bar[s], kb * BK, 0);
            }
        }
    } else if (warp == 1 && lane == 0) {
        int it = 0, local = 0;
        for (int item = blockIdx.x; item < items && ok; item += gridDim.x, ++local) {
            int kb0, kb1;
            k_range(item, kb0, kb1);
            const int acc = local & 1;
            if (!mbar_wait_suspend(&acc_empty[acc], ((local >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d = tmem + acc * TCOLS;
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int s = it % SK_STAGES;
                if (!mbar_wait_suspend(&full_bar[s], (it / SK_STAGES) & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sa = smem_u32(smem + s * SK_STAGE_BYTES);
                const uint64_t wdesc = sdesc_kmajor_sw128(sa), xdesc = sdesc_kmajor_sw128(sa + SK_W_BYTES);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    umma_bf16_ss(d, wdesc + 2 * k, xdesc + 2 * k, IDESC, (kb > kb0 || k > 0));
                umma_commit(&empty_bar[s]);
            }
            if (!ok) break;
            umma_commit(&acc_full[acc]);
        }
    } else if (warp >= 2) {
        const int quarter = warp & 3;
        int local = 0;
        for (int item = blockIdx.x; item < items; item += gridDim.x, ++local) {
            const int acc = local & 1;
            const int n = (item % row_blocks) * 128 + quarter * 32 + lane;  // weight row = TMEM lane
            const int split = item / row_blocks;
            if (!__all_sync(0xffffffffu, mbar_wait_suspend(&acc_full[acc], (local >> 1) & 1, abort_flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t v[MP];
            const uint32_t ta = tmem + ((uint32_t)(quarter * 32) << 16) + acc * TCOLS;
            if constexpr (MP == 16) {
                tmem_ld_32x32b_x16(ta, v);
            } else {
#pragma unroll
                for (int c = 0; c < MP / 32; ++c)
                    tmem_ld_32x32b_x32(ta + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[c * 32]));
            }
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&acc_empty[acc]);
            if (n < args.N) {
                if (args.splits == 1 && args.out) {
#pragma unroll
                    for (int b = 0; b < MP; ++b)
                        if (b < args.M) args.out[(size_t)b * args.ldo + n] = __uint_as_float(v[b]);
                } else {
                    float* slice = args.ws + (size_t)split * args.M * args.ldw;
#pragma unroll
                    for (int b = 0; b < MP; ++b)
                        if (b < args.M) slice[(size_t)b * args.ldw + n] = __uint_as_float(v[b]);
                }
            }
        }
    }
    if (!ok) {
        *abort_flag = 1;
        if (args.err) atomicOr(args.err, ERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 2 * TCOLS);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// EPI_RESIDUAL_NORM: one cooperative launch (all CTAs resident at once, which the row blocks' meeting
// points rely on) of a multiple of N / BN CTAs, at most one per SM.
template <int BN>
cudaError_t launch_norm(const GemmMaps& m, const GemmArgs& a, cudaStream_t st) {
    const int csize = a.N / BN, tiles = ((a.M + BM - 1) / BM) * csize;
    if (a.N % BN || csize < 1 || csize > 8 || !a.norm.gamma || !a.norm.part || !a.norm.count)
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(std::min(tiles, device_sm_count() / csize * csize));
    cfg.blockDim = dim3(EpiShape<EPI_RESIDUAL_NORM>::THREADS);
    cfg.dynamicSmemBytes = Cfg<BN>::SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gemm_tcgen05_kernel<EPI_RESIDUAL_NORM, BN>, m.a, m.b, m.c, m.r, m.v, a);
}

template <int EPI, int BN>
cudaError_t launch_epi(const GemmMaps& m, const GemmArgs& a, cudaStream_t st) {
    const int tiles = ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
    const int grid = std::min(tiles, device_sm_count());
    return launch_pdl(gemm_tcgen05_kernel<EPI, BN>, dim3(grid), dim3(EpiShape<EPI>::THREADS), Cfg<BN>::SMEM_BYTES, st,
                      m.a, m.b, m.c,
                      m.r, m.v, a);
}

}  // namespace

int device_sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (cached[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 1;
    }
    return cached[dev];
}

cudaError_t gemm_prepare() {
    cudaError_t e = cudaSuccess;
    const void* f256[] = {(const void*)gemm_tcgen05_kernel<EPI_BF16, 256>, (const void*)gemm_tcgen05_kernel<EPI_SWIGLU, 256>,
                          (const void*)gemm_tcgen05_kernel<EPI_RESIDUAL, 256>, (const void*)gemm_tcgen05_kernel<EPI_F32, 256>,
                          (const void*)gemm_tcgen05_kernel<EPI_QKV_ROPE, 256>,
                          (const void*)gemm_tcgen05_kernel<EPI_RESIDUAL_NORM, 256>};
    const void* f128[] = {(const void*)gemm_tcgen05_kernel<EPI_BF16, 128>, (const void*)gemm_tcgen05_kernel<EPI_RESIDUAL, 128>,
                          (const void*)gemm_tcgen05_kernel<EPI_F32, 128>, (const void*)gemm_tcgen05_kernel<EPI_QKV_ROPE, 128>,
                          (const void*)gemm_tcgen05_kernel<EPI_RESIDUAL_NORM, 128>};
    for (const void* f : f256) {
        cudaError_t r = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<256>::SMEM_BYTES);
        if (r != cudaSuccess) e = r;
    }
    for (const void* f : f128) {
        cudaError_t r = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<128>::SMEM_BYTES);
        if (r != cudaSuccess) e = r;
    }
    const void* fsk[] = {(const void*)gemm_skinny_kernel<16>, (const void*)gemm_skinny_kernel<32>,
                         (const void*)gemm_skinny_kernel<64>};
    for (const void* f : fsk) {
        cudaError_t r = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, SK_SMEM);
        if (r != cudaSuccess) e = r;
    }
    return e;
}

bool device_is_sm103() {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    return major == 10 && minor == 3;
}

static bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                      uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                         uint32_t box_inner, uint32_t box_outer) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, inner, outer, row_bytes, box_inner, box_outer);
}

// [d2][d1][d0] bf16 tensor, boxes of 64 x 128 x 1 in the 128-byte swizzle.
bool encode_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_out(CUtensorMap* map, const void* base, bool f32, uint64_t cols, uint64_t rows, uint64_t ld) {
    if (f32) return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, cols, rows, ld * 4, 32, kGemmBM);
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, cols, rows, ld * 2, 64, kGemmBM);
}

bool encode_gemm_maps(CUtensorMap* ta, CUtensorMap* tb, const void* A, uint64_t a_rows, const void* B, uint64_t N,
                      uint64_t K) {
    return encode_tmap_bf16_2d(ta, A, K, a_rows, K * 2, BK, BM) && encode_tmap_bf16_2d(tb, B, K, N, K * 2, BK, kGemmBoxN);
}

int gemm_tile_n(int M, int N, int epi) {
    // 128-wide tiles when 256-wide ones would leave SMs idle (SwiGLU needs the 256-wide gate|up tile)
    if (epi == EPI_SWIGLU) return 256;
    const long long tiles256 = (long long)((M + BM - 1) / BM) * ((N + 255) / 256);
    return tiles256 < device_sm_count() ? 128 : 256;
}

cudaError_t gemm_launch(const GemmMaps& m, const GemmArgs& a, cudaStream_t st) {
    if (a.M <= 0 || a.N <= 0) return cudaSuccess;
    const bool narrow = gemm_tile_n(a.M, a.N, a.epi) == 128;
    switch (a.epi) {
        case EPI_BF16: return narrow ? launch_epi<EPI_BF16, 128>(m, a, st) : launch_epi<EPI_BF16, 256>(m, a, st);
        case EPI_SWIGLU: return launch_epi<EPI_SWIGLU, 256>(m, a, st);
        case EPI_RESIDUAL: return narrow ? launch_epi<EPI_RESIDUAL, 128>(m, a, st) : launch_epi<EPI_RESIDUAL, 256>(m, a, st);
        case EPI_F32: return narrow ? launch_epi<EPI_F32, 128>(m, a, st) : launch_epi<EPI_F32, 256>(m, a, st);
        case EPI_QKV_ROPE: return narrow ? launch_epi<EPI_QKV_ROPE, 128>(m, a, st) : launch_epi<EPI_QKV_ROPE, 256>(m, a, st);
        case EPI_RESIDUAL_NORM: return narrow ? launch_norm<128>(m, a, st) : launch_norm<256>(m, a, st);
    }
    return cudaErrorInvalidValue;
}

bool gemm_norm_fusable(int M, int N) {
    const int bn = gemm_tile_n(M, N, EPI_RESIDUAL_NORM);
    return M > 0 && N % bn == 0 && N / bn <= 8;
}

bool gemm_norm_preferred(int M, int N) {
    // With the eight-warp epilogue the row block's meeting costs less than the separate RMSNorm pass at
    // every measured size (0.6B: 2048 rows 2.83 -> 2.79 ms per prefill step; 32768 rows 118 -> 112 us
    // per o_proj and norm).
    return gemm_norm_fusable(M, N);
}

size_t gemm_norm_part_floats(int M) { return (size_t)((M + BM - 1) / BM) * 8 * 2 * BM; }
size_t gemm_norm_count_ints(int M) { return (size_t)((M + BM - 1) / BM) * 2; }

bool encode_skinny_x_map(CUtensorMap* map, const void* X, uint64_t rows, uint64_t K) {
    return encode_tmap_bf16_2d(map, X, K, rows, K * 2, BK, kSkinnyRowsBox);
}

int skinny_splits(int N, int K) {
    // The persistent kernel spreads tiles x splits items over the SMs; its time goes as the items of the
    // busiest CTA times the K blocks of an item, plus the slices the finalize step reads back (counted
    // for 64 rows, in 16-KB weight-block units per SM). Take the split count (<= 16, >= 2 K blocks per
    // item) that minimises the sum, the fewest splits among equals.
    const int tiles = (N + 127) / 128, k_blocks = (K + BK - 1) / BK, sms = device_sm_count();
    int best = 1;
    long long best_cost = -1;
    for (int s = 1; s <= 16 && (s == 1 || k_blocks / s >= 2); ++s) {
        const int per = (k_blocks + s - 1) / s;
        const int used = (k_blocks + per - 1) / per;  // no empty splits
        if (used != s) continue;
        const long long rounds = ((long long)tiles * s + sms - 1) / sms;
        const double slices = (double)s * kSkinnyRowsBox * N * 4 / ((double)sms * 128 * BK * 2);
        const long long cost = rounds * per + (long long)(slices + 0.5);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

cudaError_t gemm_skinny_launch(const CUtensorMap& tw, const CUtensorMap& tx, const SkinnyArgs& a, cudaStream_t st) {
    if (a.M <= 0 || a.N <= 0) return cudaSuccess;
    if (a.M > kSkinnyRowsBox) return cudaErrorInvalidValue;
    const int items = (a.N + 127) / 128 * a.splits;
    const dim3 grid(std::min(items, device_sm_count()));
    if (a.M <= 16) return launch_pdl(gemm_skinny_kernel<16>, grid, dim3(THREADS), SK_SMEM, st, tw, tx, a);
    if (a.M <= 32) return launch_pdl(gemm_skinny_kernel<32>, grid, dim3(THREADS), SK_SMEM, st, tw, tx, a);
    return launch_pdl(gemm_skinny_kernel<64>, grid, dim3(THREADS), SK_SMEM, st, tw, tx, a);
}

}  // namespace q3
