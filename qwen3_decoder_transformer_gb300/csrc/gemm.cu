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
// Design (sm_103a): a persistent kernel, one CTA per SM, 6 warps.
//   warp 0      TMA producer: 128x64 A and 256x64 B boxes (128-byte swizzle) into a 4-stage ring.
//   warp 1      TMEM owner and MMA issuer: one thread issues tcgen05.mma 128x256x16 (4 per stage)
//               into one of two 256-column fp32 accumulators, and commits stage releases and
//               accumulator-ready signals to mbarriers.
//   warps 2-5   epilogue: tcgen05.ld of the accumulator rows (warp w reads TMEM lanes 32*(w%4)..),
//               fused epilogue math, 16-byte global stores; then release the accumulator.
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
constexpr int THREADS = 192;
// Per tile width BN (256, or 128 when 256-wide tiles cannot fill the SMs): stage size, ring depth,
// TMEM columns (two accumulators) and the instruction descriptor.
template <int BN>
struct Cfg {
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = BN == 256 ? 4 : 6;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
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
template <int DH, int BN>
__device__ __forceinline__ void epilogue_qkv_rope(const GemmArgs& a, uint32_t tacc, int row, int n0) {
    const QkvRopeArgs& q = a.qkv;
    const bool row_ok = row < a.M;
    const int b = row_ok ? row / q.T : 0, t = row_ok ? row % q.T : 0;
    const int pos = *q.len0 + t;
    constexpr int HALF = DH / 2;
#pragma unroll 1
    for (int lh = 0; lh < BN / DH; ++lh) {
        const int hg = n0 / DH + lh;
        const uint32_t th = tacc + lh * DH;
        if (hg >= q.Hq + q.Hkv) {  // V head: copy to the cache slot
            __nv_bfloat16* dst = q.v_cache + (((size_t)b * q.Hkv + (hg - q.Hq - q.Hkv)) * q.cap + pos) * DH;
#pragma unroll 1
            for (int c = 0; c < DH / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(th + c * 32, r);
                tmem_ld_wait();
                if (!row_ok) continue;
                uint32_t w[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) w[j] = pack_bf16(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    reinterpret_cast<uint4*>(dst + c * 32)[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
            }
            continue;
        }
        const bool is_q = hg < q.Hq;
        // pass 1: sum of squares of the bf16-rounded projection
        float ss = 0.f;
#pragma unroll 1
        for (int c = 0; c < DH / 32; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(th + c * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float x = rbf(__uint_as_float(r[j]));
                ss = fmaf(x, x, ss);
            }
        }
        const float rn = __frsqrt_rn(ss / (float)DH + q.eps);
        const __nv_bfloat16* gam = is_q ? q.q_gamma : q.k_gamma;
        const __nv_bfloat16* cs = q.table + (size_t)pos * DH;
        __nv_bfloat16* dst = is_q ? q.q_out + (((size_t)b * q.Hq + hg) * q.T + t) * DH
                                  : q.k_cache + (((size_t)b * q.Hkv + (hg - q.Hq)) * q.cap + pos) * DH;
        // pass 2: 32 rotation pairs at a time, (i, i + HALF)
#pragma unroll 1
        for (int c = 0; c < HALF / 32; ++c) {
            uint32_t lo[32], hi[32];
            tmem_ld_32x32b_x32(th + c * 32, lo);
            tmem_ld_32x32b_x32(th + HALF + c * 32, hi);
            tmem_ld_wait();
            if (!row_ok) continue;
            uint32_t wlo[16], whi[16];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 g0 = __ldg(reinterpret_cast<const uint4*>(gam + c * 32) + v);
                const uint4 g1 = __ldg(reinterpret_cast<const uint4*>(gam + HALF + c * 32) + v);
                const uint4 cc = __ldg(reinterpret_cast<const uint4*>(cs + c * 32) + v);
                const uint4 sn = __ldg(reinterpret_cast<const uint4*>(cs + HALF + c * 32) + v);
                const uint32_t G0[4] = {g0.x, g0.y, g0.z, g0.w}, G1[4] = {g1.x, g1.y, g1.z, g1.w};
                const uint32_t C[4] = {cc.x, cc.y, cc.z, cc.w}, S[4] = {sn.x, sn.y, sn.z, sn.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float o_lo[2], o_hi[2];
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int j = 8 * v + 2 * e + k;
                        const float ga = k ? bf16_hi(G0[e]) : bf16_lo(G0[e]);
                        const float gb = k ? bf16_hi(G1[e]) : bf16_lo(G1[e]);
                        const float co = k ? bf16_hi(C[e]) : bf16_lo(C[e]);
                        const float si = k ? bf16_hi(S[e]) : bf16_lo(S[e]);
                        const float av = rbf(ga * rbf(rbf(__uint_as_float(lo[j])) * rn));
                        const float bv = rbf(gb * rbf(rbf(__uint_as_float(hi[j])) * rn));
                        o_lo[k] = rbf(av * co) + rbf(-(bv * si));
                        o_hi[k] = rbf(bv * co) + rbf(av * si);
                    }
                    wlo[4 * v + e] = pack_bf16(o_lo[0], o_lo[1]);
                    whi[4 * v + e] = pack_bf16(o_hi[0], o_hi[1]);
                }
            }
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                reinterpret_cast<uint4*>(dst + c * 32)[v] = make_uint4(wlo[4 * v], wlo[4 * v + 1], wlo[4 * v + 2], wlo[4 * v + 3]);
                reinterpret_cast<uint4*>(dst + HALF + c * 32)[v] =
                    make_uint4(whi[4 * v], whi[4 * v + 1], whi[4 * v + 2], whi[4 * v + 3]);
            }
        }
    }
}

template <int EPI, int BN>
__device__ __forceinline__ void epilogue_chunks(const GemmArgs& a, uint32_t tacc, int row, int n0) {
    const bool row_ok = row < a.M;
    if constexpr (EPI == EPI_QKV_ROPE) {
        if (a.qkv.dh == 128) epilogue_qkv_rope<128, BN>(a, tacc, row, n0);
        else epilogue_qkv_rope<64, BN>(a, tacc, row, n0);
    } else if constexpr (EPI == EPI_SWIGLU) {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.C) + (size_t)row * a.ldc + n0 / 2;
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
            uint32_t g[32], u[32];
            tmem_ld_32x32b_x32(tacc + c * 32, g);
            tmem_ld_32x32b_x32(tacc + BN / 2 + c * 32, u);
            tmem_ld_wait();
            if (!row_ok) continue;
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                float g0 = rbf(__uint_as_float(g[2 * j])), g1 = rbf(__uint_as_float(g[2 * j + 1]));
                float s0 = rbf(g0 / (1.0f + expf(-g0))), s1 = rbf(g1 / (1.0f + expf(-g1)));
                w[j] = pack_bf16(s0 * rbf(__uint_as_float(u[2 * j])), s1 * rbf(__uint_as_float(u[2 * j + 1])));
            }
            uint4* dst = reinterpret_cast<uint4*>(out + c * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
        }
    } else {
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(tacc + c * 32, r);
            tmem_ld_wait();
            const int col0 = n0 + c * 32;
            if (!row_ok || col0 >= a.N) continue;
            const bool full = col0 + 32 <= a.N;
            if constexpr (EPI == EPI_F32) {
                float* dst = reinterpret_cast<float*>(a.C) + (size_t)row * a.ldc + col0;
                if (full) {
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        reinterpret_cast<float4*>(dst)[v] =
                            make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                        __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
                } else {
                    for (int j = 0; j < a.N - col0; ++j) dst[j] = __uint_as_float(r[j]);
                }
            } else {
                __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.C) + (size_t)row * a.ldc + col0;
                float add[32];
                if constexpr (EPI == EPI_RESIDUAL) {
                    const __nv_bfloat16* src = a.R + (size_t)row * a.ldr + col0;
                    if (full) {
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint4 q = reinterpret_cast<const uint4*>(src)[v];
                            uint32_t qq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                add[8 * v + 2 * e] = bf16_lo(qq[e]);
                                add[8 * v + 2 * e + 1] = bf16_hi(qq[e]);
                            }
                        }
                    } else {
                        for (int j = 0; j < 32; ++j) add[j] = (col0 + j < a.N) ? bf16f(src[j]) : 0.f;
                    }
                }
                uint32_t w[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float x0 = __uint_as_float(r[2 * j]), x1 = __uint_as_float(r[2 * j + 1]);
                    if constexpr (EPI == EPI_RESIDUAL) {
                        x0 = add[2 * j] + rbf(x0);
                        x1 = add[2 * j + 1] + rbf(x1);
                    }
                    w[j] = pack_bf16(x0, x1);
                }
                if (full) {
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        reinterpret_cast<uint4*>(dst)[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
                } else {
                    for (int j = 0; j < a.N - col0; ++j) {
                        uint32_t h = (j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xffffu);
                        reinterpret_cast<uint16_t*>(dst)[j] = (uint16_t)h;
                    }
                }
            }
        }
    }
}

template <int EPI, int BN>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const GemmArgs args) {
    using C = Cfg<BN>;
    constexpr int STAGES = C::STAGES, STAGE_BYTES = C::STAGE_BYTES, TMEM_COLS = C::TMEM_COLS;
    constexpr uint32_t IDESC = C::IDESC;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    uint64_t* empty_bar = full_bar + STAGES;
    uint64_t* acc_full = empty_bar + STAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tiles = (args.M + BM - 1) / BM, n_tiles = (args.N + BN - 1) / BN;
    const int k_blocks = (args.K + BK - 1) / BK;
    const int total = m_tiles * n_tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 128);
        }
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
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
    pdl_wait();  // inputs of this GEMM come from the previous kernel
    pdl_trigger();

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer
        int it = 0;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const Tile tl = tile_of<BN>(t, m_tiles, n_tiles);
            for (int kb = 0; kb < k_blocks; ++kb, ++it) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1;
                if (!mbar_wait(&empty_bar[s], ph ^ 1, abort_flag)) { ok = false; break; }
                uint8_t* sa = smem + s * STAGE_BYTES;
                mbar_expect_tx(&full_bar[s], STAGE_BYTES);
                tma_load_2d(sa, &tmA, &full_bar[s], kb * BK, tl.m0);
#pragma unroll
                for (int nb = 0; nb < BN / kGemmBoxN; ++nb)
                    tma_load_2d(sa + A_BYTES + nb * kGemmBoxN * BK * 2, &tmB, &full_bar[s], kb * BK, tl.n0 + nb * kGemmBoxN);
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        int it = 0, local = 0;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++local) {
            const int acc = local & 1;
            const uint32_t aph = (local >> 1) & 1;
            if (!mbar_wait(&acc_empty[acc], aph ^ 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * BN;
            for (int kb = 0; kb < k_blocks; ++kb, ++it) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1;
                if (!mbar_wait(&full_bar[s], ph, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sa = smem_u32(smem + s * STAGE_BYTES);
                const uint64_t adesc = sdesc_kmajor_sw128(sa), bdesc = sdesc_kmajor_sw128(sa + A_BYTES);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    umma_bf16_ss(d_tmem, adesc + 2 * k, bdesc + 2 * k, IDESC, (kb | k) != 0);
                umma_commit(&empty_bar[s]);
            }
            if (!ok) break;
            umma_commit(&acc_full[acc]);
        }
    } else if (warp >= 2) {
        // ---------------- epilogue
        const int quarter = warp & 3;
        int local = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++local) {
            const int acc = local & 1;
            const uint32_t aph = (local >> 1) & 1;
            // every lane waits, so the warp stays converged for the .sync.aligned TMEM loads
            if (!mbar_wait(&acc_full[acc], aph, abort_flag)) { ok = false; }
            if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
            tc_fence_after();
            const Tile tl = tile_of<BN>(t, m_tiles, n_tiles);
            const uint32_t tacc = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
            epilogue_chunks<EPI, BN>(args, tacc, tl.m0 + quarter * 32 + lane, tl.n0);
            tc_fence_before();
            mbar_arrive(&acc_empty[acc]);
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
        tmem_dealloc(tmem_base, TMEM_COLS);
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

template <int EPI, int BN>
cudaError_t launch_epi(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a, cudaStream_t st) {
    const int tiles = ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
    const int grid = std::min(tiles, device_sm_count());
    return launch_pdl(gemm_tcgen05_kernel<EPI, BN>, dim3(grid), dim3(THREADS), Cfg<BN>::SMEM_BYTES, st, ta, tb, a);
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
                          (const void*)gemm_tcgen05_kernel<EPI_QKV_ROPE, 256>};
    const void* f128[] = {(const void*)gemm_tcgen05_kernel<EPI_BF16, 128>, (const void*)gemm_tcgen05_kernel<EPI_RESIDUAL, 128>,
                          (const void*)gemm_tcgen05_kernel<EPI_F32, 128>, (const void*)gemm_tcgen05_kernel<EPI_QKV_ROPE, 128>};
    for (const void* f : f256) {
        cudaError_t r = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<256>::SMEM_BYTES);
        if (r != cudaSuccess) e = r;
    }
    for (const void* f : f128) {
        cudaError_t r = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<128>::SMEM_BYTES);
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

bool encode_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                         uint32_t box_inner, uint32_t box_outer) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
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

cudaError_t gemm_launch(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& a, cudaStream_t st) {
    if (a.M <= 0 || a.N <= 0) return cudaSuccess;
    const bool narrow = gemm_tile_n(a.M, a.N, a.epi) == 128;
    switch (a.epi) {
        case EPI_BF16: return narrow ? launch_epi<EPI_BF16, 128>(ta, tb, a, st) : launch_epi<EPI_BF16, 256>(ta, tb, a, st);
        case EPI_SWIGLU: return launch_epi<EPI_SWIGLU, 256>(ta, tb, a, st);
        case EPI_RESIDUAL:
            return narrow ? launch_epi<EPI_RESIDUAL, 128>(ta, tb, a, st) : launch_epi<EPI_RESIDUAL, 256>(ta, tb, a, st);
        case EPI_F32: return narrow ? launch_epi<EPI_F32, 128>(ta, tb, a, st) : launch_epi<EPI_F32, 256>(ta, tb, a, st);
        case EPI_QKV_ROPE:
            return narrow ? launch_epi<EPI_QKV_ROPE, 128>(ta, tb, a, st) : launch_epi<EPI_QKV_ROPE, 256>(ta, tb, a, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace q3
