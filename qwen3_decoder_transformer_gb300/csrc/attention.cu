// Causal grouped-query attention over the KV cache ("A modern architecture: Qwen3", Attention with
// grouped KV heads and Q/K normalization; "Transformer architectures: modern", section 3: query head
// h reads kv head floor(h / g), g = Hq / Hkv; scores scaled by head_dim^-0.5; causal mask).
//
// Prefill: flash attention with an online softmax. A CTA owns 64 query rows of one (sequence,
// query head); four warps each own 16 rows. K/V tiles of 64 keys stream through a double-buffered,
// XOR-swizzled shared-memory ring (cp.async); S = Q K^T and O += P V run on the tensor cores
// (mma.m16n8k16 bf16, fp32 accumulate); P stays in registers as bf16. Tiles above the diagonal are
// skipped; query tiles are scheduled longest-first.
//
// Decode: one query per (sequence, query head) against the whole cache. A CTA owns a 256-key
// chunk of one (sequence, kv head) and serves all g query heads of that group from one read of
// K and V (16-byte coalesced loads, 8 in flight per thread). Partial (max, sum, output) triples
// go to a workspace; a second kernel merges the chunks by log-sum-exp.
#include <cfloat>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace q3 {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk `c` of row `r` in a tile whose rows are CH chunks wide, XOR-swizzled
// on the low three bits so that 8 consecutive rows at one logical chunk hit 8 different banks.
template <int CH>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return (uint32_t)(r * CH * 16 + ((c ^ (r & 7)) * 16));
}

constexpr int FA_BQ = 64, FA_BKV = 64, FA_THREADS = 128;

template <int DH>
__global__ void __launch_bounds__(FA_THREADS)
    attn_prefill_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kc,
                        const __nv_bfloat16* __restrict__ vc, int T, int Hq, int Hkv, int cap,
                        const int* __restrict__ len0p, __nv_bfloat16* __restrict__ out) {
    constexpr int CH = DH / 8;  // 16-byte chunks per row
    constexpr int TILE_BYTES = FA_BKV * DH * 2;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* sQ = smem;
    uint8_t* sK = smem + FA_BQ * DH * 2;  // 2 stages
    uint8_t* sV = sK + 2 * TILE_BYTES;    // 2 stages

    const int qt = gridDim.x - 1 - blockIdx.x;  // longest (highest) query tiles first
    const int h = blockIdx.y, b = blockIdx.z;
    const int j = h / (Hq / Hkv);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int len0 = *len0p;
    const int q_begin = qt * FA_BQ;
    const int q_end = min(T, q_begin + FA_BQ);
    const int n_valid = len0 + q_end;  // keys 0 .. n_valid-1 may be visible to this tile
    const int n_tiles = (n_valid + FA_BKV - 1) / FA_BKV;

    const __nv_bfloat16* qb = q + (((size_t)b * Hq + h) * T) * DH;
    const __nv_bfloat16* kb = kc + (((size_t)b * Hkv + j) * cap) * DH;
    const __nv_bfloat16* vb = vc + (((size_t)b * Hkv + j) * cap) * DH;

    // Q tile (rows past T are zero-filled)
    for (int i = threadIdx.x; i < FA_BQ * CH; i += FA_THREADS) {
        const int r = i / CH, c = i % CH;
        const int t = q_begin + r;
        cp_async16(smem_u32(sQ) + swz<CH>(r, c), qb + (size_t)min(t, T - 1) * DH + c * 8, t < T ? 16 : 0);
    }
    auto load_kv = [&](int tile, int stage) {
        const int k0 = tile * FA_BKV;
        for (int i = threadIdx.x; i < FA_BKV * CH; i += FA_THREADS) {
            const int r = i / CH, c = i % CH;
            const int s = k0 + r;
            const int nb = s < n_valid ? 16 : 0;
            const size_t off = (size_t)min(s, n_valid - 1) * DH + c * 8;
            cp_async16(smem_u32(sK + stage * TILE_BYTES) + swz<CH>(r, c), kb + off, nb);
            cp_async16(smem_u32(sV + stage * TILE_BYTES) + swz<CH>(r, c), vb + off, nb);
        }
    };
    load_kv(0, 0);
    cp_async_commit();

    // per-thread rows: g = lane/4 and g+8 within the warp's 16 rows
    const int g = lane >> 2, cq = lane & 3;
    const int row0 = q_begin + warp * 16 + g, row1 = row0 + 8;
    const int p0 = len0 + row0, p1 = len0 + row1;  // absolute positions
    const float sl2 = kLog2e / sqrtf((float)DH);

    uint32_t qf[DH / 16][4];
    float o[DH / 8][4];
#pragma unroll
    for (int n = 0; n < DH / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int tile = 0; tile < n_tiles; ++tile) {
        const int stage = tile & 1;
        if (tile + 1 < n_tiles) load_kv(tile + 1, stage ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (tile == 0) {
#pragma unroll
            for (int kk = 0; kk < DH / 16; ++kk) {
                const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = kk * 2 + (lane >> 4);
                ldmatrix_x4(smem_u32(sQ) + swz<CH>(r, c), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
            }
        }
        const uint32_t kbase = smem_u32(sK + stage * TILE_BYTES), vbase = smem_u32(sV + stage * TILE_BYTES);
        // S = Q K^T for 64 keys: 8 n-tiles of 8 keys
        float s[FA_BKV / 8][4];
#pragma unroll
        for (int n = 0; n < FA_BKV / 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
#pragma unroll
            for (int np = 0; np < FA_BKV / 16; ++np) {
                const int r = np * 16 + (lane & 7) + (lane >> 4) * 8;
                const int c = kk * 2 + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(kbase + swz<CH>(r, c), b0, b1, b2, b3);
                mma_bf16_16816(s[2 * np], qf[kk], b0, b1);
                mma_bf16_16816(s[2 * np + 1], qf[kk], b2, b3);
            }
        }
        // causal mask where the tile reaches past the first row's position
        const int k0 = tile * FA_BKV;
        if (k0 + FA_BKV - 1 > len0 + q_begin) {
#pragma unroll
            for (int n = 0; n < FA_BKV / 8; ++n) {
                const int key = k0 + n * 8 + 2 * cq;
                if (key > p0 || key >= n_valid) s[n][0] = -INFINITY;
                if (key + 1 > p0 || key + 1 >= n_valid) s[n][1] = -INFINITY;
                if (key > p1 || key >= n_valid) s[n][2] = -INFINITY;
                if (key + 1 > p1 || key + 1 >= n_valid) s[n][3] = -INFINITY;
            }
        }
        // online softmax (base 2): rows g (s[.][0..1]) and g+8 (s[.][2..3])
        float mx0 = m0, mx1 = m1;
#pragma unroll
        for (int n = 0; n < FA_BKV / 8; ++n) {
            mx0 = fmaxf(mx0, fmaxf(s[n][0], s[n][1]) * sl2);
            mx1 = fmaxf(mx1, fmaxf(s[n][2], s[n][3]) * sl2);
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float c0 = exp2f(m0 - mx0), c1 = exp2f(m1 - mx1);  // m = -inf initially -> 0
        m0 = mx0;
        m1 = mx1;
        float rs0 = 0.f, rs1 = 0.f;
        uint32_t pf[FA_BKV / 16][4];
#pragma unroll
        for (int n = 0; n < FA_BKV / 8; ++n) {
            const float e0 = exp2f(s[n][0] * sl2 - mx0), e1 = exp2f(s[n][1] * sl2 - mx0);
            const float e2 = exp2f(s[n][2] * sl2 - mx1), e3 = exp2f(s[n][3] * sl2 - mx1);
            rs0 += e0 + e1;
            rs1 += e2 + e3;
            pf[n / 2][(n & 1) * 2 + 0] = pack_bf16(e0, e1);
            pf[n / 2][(n & 1) * 2 + 1] = pack_bf16(e2, e3);
        }
        l0 = l0 * c0 + rs0;
        l1 = l1 * c1 + rs1;
#pragma unroll
        for (int n = 0; n < DH / 8; ++n) {
            o[n][0] *= c0;
            o[n][1] *= c0;
            o[n][2] *= c1;
            o[n][3] *= c1;
        }
        // O += P V: k-steps of 16 keys, n-tiles of 8 head features
#pragma unroll
        for (int kk = 0; kk < FA_BKV / 16; ++kk) {
            const uint32_t a[4] = {pf[kk][0], pf[kk][1], pf[kk][2], pf[kk][3]};
#pragma unroll
            for (int np = 0; np < DH / 16; ++np) {
                const int r = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = np * 2 + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4_trans(vbase + swz<CH>(r, c), b0, b1, b2, b3);
                mma_bf16_16816(o[2 * np], a, b0, b1);
                mma_bf16_16816(o[2 * np + 1], a, b2, b3);
            }
        }
        __syncthreads();  // the stage is reloaded next iteration
    }
    cp_async_wait<0>();

    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float inv0 = 1.f / l0, inv1 = 1.f / l1;
    const size_t ld = (size_t)Hq * DH;
    __nv_bfloat16* ob = out + ((size_t)b * T) * ld + (size_t)h * DH;
#pragma unroll
    for (int n = 0; n < DH / 8; ++n) {
        const int col = n * 8 + 2 * cq;
        if (row0 < T)
            *reinterpret_cast<uint32_t*>(ob + (size_t)row0 * ld + col) = pack_bf16(o[n][0] * inv0, o[n][1] * inv0);
        if (row1 < T)
            *reinterpret_cast<uint32_t*>(ob + (size_t)row1 * ld + col) = pack_bf16(o[n][2] * inv1, o[n][3] * inv1);
    }
}

// ------------------------------------------------------------------------------------- decode
constexpr int DEC_CHUNK = 256, DEC_THREADS = 128, DEC_UNROLL = 8;

__device__ __forceinline__ int dec_splits(int cap) { return (cap + DEC_CHUNK - 1) / DEC_CHUNK; }

// Workspace layout per (b, q-head, split): [m, l] floats, then DH floats of unnormalised output.
template <int DH, int G>
__global__ void __launch_bounds__(DEC_THREADS)
    attn_decode_split_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kc,
                             const __nv_bfloat16* __restrict__ vc, int Hq, int Hkv, int cap,
                             const int* __restrict__ len0p, float* __restrict__ work) {
    constexpr int LPK = DH / 8;   // lanes per key row (16-byte pieces)
    constexpr int KPW = 32 / LPK;  // keys per warp per step
    constexpr int KPS = KPW * (DEC_THREADS / 32);  // keys per block step
    constexpr int REC = DH + 2;
    __shared__ float sc[G][DEC_CHUNK];
    __shared__ float red[DEC_THREADS / 32][G][DH];
    __shared__ float stat[G][2];

    const int split = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
    const int nsplit = gridDim.x;
    const int n = *len0p + 1;
    const int s0 = split * DEC_CHUNK, s1 = min(n, s0 + DEC_CHUNK);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane / LPK, li = lane % LPK;
    float* wb = work + (((size_t)b * Hq + (size_t)j * G) * nsplit + split) * REC;
    if (s0 >= n) {
        if (threadIdx.x < G) {
            wb[(size_t)threadIdx.x * nsplit * REC + 0] = -INFINITY;
            wb[(size_t)threadIdx.x * nsplit * REC + 1] = 0.f;
        }
        return;
    }
    const size_t kvbase = (((size_t)b * Hkv + j) * cap) * DH;
    const float sl2 = kLog2e / sqrtf((float)DH);
    float qv[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const uint4 v = *reinterpret_cast<const uint4*>(q + ((size_t)b * Hq + (size_t)j * G + h) * DH + li * 8);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            qv[h][2 * e] = bf16_lo(w[e]) * sl2;
            qv[h][2 * e + 1] = bf16_hi(w[e]) * sl2;
        }
    }
    // pass 1: scores (already in log2 units)
    for (int base = s0; base < s1; base += KPS * DEC_UNROLL) {
        uint4 kv[DEC_UNROLL];
#pragma unroll
        for (int u = 0; u < DEC_UNROLL; ++u) {
            const int s = base + u * KPS + warp * KPW + sub;
            kv[u] = s < s1 ? *reinterpret_cast<const uint4*>(kc + kvbase + (size_t)s * DH + li * 8)
                           : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < DEC_UNROLL; ++u) {
            const int s = base + u * KPS + warp * KPW + sub;
            const uint32_t w[4] = {kv[u].x, kv[u].y, kv[u].z, kv[u].w};
            float d[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float acc = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc = fmaf(qv[h][2 * e], bf16_lo(w[e]), acc);
                    acc = fmaf(qv[h][2 * e + 1], bf16_hi(w[e]), acc);
                }
#pragma unroll
                for (int o = LPK / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                d[h] = acc;
            }
            if (li == 0 && s < s1) {
#pragma unroll
                for (int h = 0; h < G; ++h) sc[h][s - s0] = d[h];
            }
        }
    }
    __syncthreads();
    // chunk max and exponentials, one warp per head
    const int cnt = s1 - s0;
    for (int h = warp; h < G; h += DEC_THREADS / 32) {
        float mx = -INFINITY;
        for (int i = lane; i < cnt; i += 32) mx = fmaxf(mx, sc[h][i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float sum = 0.f;
        for (int i = lane; i < cnt; i += 32) {
            const float e = exp2f(sc[h][i] - mx);
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
    __syncthreads();
    // pass 2: weighted sum of V rows
    float acc[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[h][e] = 0.f;
    for (int base = s0; base < s1; base += KPS * DEC_UNROLL) {
        uint4 vv[DEC_UNROLL];
#pragma unroll
        for (int u = 0; u < DEC_UNROLL; ++u) {
            const int s = base + u * KPS + warp * KPW + sub;
            vv[u] = s < s1 ? *reinterpret_cast<const uint4*>(vc + kvbase + (size_t)s * DH + li * 8)
                           : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < DEC_UNROLL; ++u) {
            const int s = base + u * KPS + warp * KPW + sub;
            if (s >= s1) continue;
            const uint32_t w[4] = {vv[u].x, vv[u].y, vv[u].z, vv[u].w};
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float p = sc[h][s - s0];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc[h][2 * e] = fmaf(p, bf16_lo(w[e]), acc[h][2 * e]);
                    acc[h][2 * e + 1] = fmaf(p, bf16_hi(w[e]), acc[h][2 * e + 1]);
                }
            }
        }
    }
    // reduce over the KPW key slots in the warp, then over warps
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float v = acc[h][e];
#pragma unroll
            for (int o = LPK; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            acc[h][e] = v;
        }
    if (sub == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < 8; ++e) red[warp][h][li * 8 + e] = acc[h][e];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < G * DH; i += DEC_THREADS) {
        const int h = i / DH, d = i % DH;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < DEC_THREADS / 32; ++w) v += red[w][h][d];
        float* rec = wb + (size_t)h * nsplit * REC;
        rec[2 + d] = v;
        if (d == 0) {
            rec[0] = stat[h][0];
            rec[1] = stat[h][1];
        }
    }
}

// Merge the chunks of one (b, q-head): O = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i.
template <int DH>
__global__ void attn_decode_combine_kernel(const float* __restrict__ work, int Hq, int nsplit,
                                           __nv_bfloat16* __restrict__ out) {
    constexpr int REC = DH + 2;
    const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
    const float* wb = work + ((size_t)b * Hq + h) * nsplit * REC;
    float M = -INFINITY;
    for (int i = 0; i < nsplit; ++i) M = fmaxf(M, wb[(size_t)i * REC]);
    float L = 0.f, acc = 0.f;
    for (int i = 0; i < nsplit; ++i) {
        const float mi = wb[(size_t)i * REC];
        if (mi == -INFINITY) continue;
        const float f = exp2f(mi - M);
        L = fmaf(wb[(size_t)i * REC + 1], f, L);
        acc = fmaf(wb[(size_t)i * REC + 2 + d], f, acc);
    }
    out[((size_t)b * Hq + h) * DH + d] = __float2bfloat16_rn(acc / L);
}

template <int DH, int G>
cudaError_t decode_launch_t(const __nv_bfloat16* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc, int B, int Hq,
                            int Hkv, int cap, const int* len0, float* work, __nv_bfloat16* out, cudaStream_t st) {
    const int nsplit = (cap + DEC_CHUNK - 1) / DEC_CHUNK;
    attn_decode_split_kernel<DH, G><<<dim3(nsplit, Hkv, B), DEC_THREADS, 0, st>>>(q, kc, vc, Hq, Hkv, cap, len0, work);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    attn_decode_combine_kernel<DH><<<dim3(Hq, B), DH, 0, st>>>(work, Hq, nsplit, out);
    return cudaGetLastError();
}

template <int DH>
cudaError_t decode_launch_dh(const __nv_bfloat16* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc, int B, int Hq,
                             int Hkv, int cap, const int* len0, float* work, __nv_bfloat16* out, cudaStream_t st) {
    switch (Hq / Hkv) {
        case 1: return decode_launch_t<DH, 1>(q, kc, vc, B, Hq, Hkv, cap, len0, work, out, st);
        case 2: return decode_launch_t<DH, 2>(q, kc, vc, B, Hq, Hkv, cap, len0, work, out, st);
        case 4: return decode_launch_t<DH, 4>(q, kc, vc, B, Hq, Hkv, cap, len0, work, out, st);
        case 8: return decode_launch_t<DH, 8>(q, kc, vc, B, Hq, Hkv, cap, len0, work, out, st);
    }
    return cudaErrorInvalidValue;
}

template <int DH>
cudaError_t prefill_launch_dh(const __nv_bfloat16* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc, int B, int T,
                              int Hq, int Hkv, int cap, const int* len0, __nv_bfloat16* out, cudaStream_t st) {
    constexpr int smem = FA_BQ * DH * 2 + 4 * FA_BKV * DH * 2;
    dim3 grid((T + FA_BQ - 1) / FA_BQ, Hq, B);
    attn_prefill_kernel<DH><<<grid, FA_THREADS, smem, st>>>(q, kc, vc, T, Hq, Hkv, cap, len0, out);
    return cudaGetLastError();
}

}  // namespace

cudaError_t attn_prefill_launch(const __nv_bfloat16* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc, int B, int T,
                                int Hq, int Hkv, int dh, int cap, const int* len0, __nv_bfloat16* out,
                                cudaStream_t st) {
    if (B <= 0 || T <= 0) return cudaSuccess;
    if (dh == 128) return prefill_launch_dh<128>(q, kc, vc, B, T, Hq, Hkv, cap, len0, out, st);
    if (dh == 64) return prefill_launch_dh<64>(q, kc, vc, B, T, Hq, Hkv, cap, len0, out, st);
    return cudaErrorInvalidValue;
}

size_t attn_decode_workspace(int B, int Hq, int dh, int cap) {
    const size_t nsplit = (size_t)(cap + DEC_CHUNK - 1) / DEC_CHUNK;
    return (size_t)B * Hq * nsplit * (dh + 2) * sizeof(float);
}

cudaError_t attn_decode_launch(const __nv_bfloat16* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc, int B, int Hq,
                               int Hkv, int dh, int cap, const int* len0, float* work, __nv_bfloat16* out,
                               cudaStream_t st) {
    if (B <= 0) return cudaSuccess;
    if (dh == 128) return decode_launch_dh<128>(q, kc, vc, B, Hq, Hkv, cap, len0, work, out, st);
    if (dh == 64) return decode_launch_dh<64>(q, kc, vc, B, Hq, Hkv, cap, len0, work, out, st);
    return cudaErrorInvalidValue;
}

int attn_decode_kernel_count() { return 2; }

cudaError_t attention_prepare() {
    cudaError_t e1 = cudaFuncSetAttribute(attn_prefill_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          FA_BQ * 128 * 2 + 4 * FA_BKV * 128 * 2);
    cudaError_t e2 = cudaFuncSetAttribute(attn_prefill_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          FA_BQ * 64 * 2 + 4 * FA_BKV * 64 * 2);
    return e1 != cudaSuccess ? e1 : e2;
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
