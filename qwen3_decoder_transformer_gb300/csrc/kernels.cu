#include <algorithm>
// Memory-bound kernels of the Qwen3 block: embedding gather, RMSNorm, the RoPE table, and the
// fused q_norm/k_norm + RoPE + KV-cache append. Each reads and writes its rows once with 8- or
// 16-byte vector accesses; one warp owns one row or one head vector.
#include "common.cuh"
#include "internal.h"

namespace q3 {
namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// x = E[ids] ("A modern architecture: Qwen3", The whole model: embed_tokens(ids)). One warp per row.
__global__ void embed_kernel(const __nv_bfloat16* __restrict__ E, int V, int d, const int32_t* __restrict__ ids, int M,
                             __nv_bfloat16* __restrict__ out, int* err) {
    pdl_wait();
    pdl_trigger();
    const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= M) return;
    const int id = ids[row];
    uint4* dst = reinterpret_cast<uint4*>(out + (size_t)row * d);
    const int nv = d / 8;
    if (id < 0 || id >= V) {
        for (int v = lane; v < nv; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
        if (lane == 0 && err) atomicOr(err, ERR_TOKEN);
        return;
    }
    const uint4* src = reinterpret_cast<const uint4*>(E + (size_t)id * d);
    for (int v = lane; v < nv; v += 32) dst[v] = __ldg(src + v);
}

__device__ __forceinline__ float sumsq8(uint4 v) {
    float s = 0.f;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float a = bf16_lo(w[e]), b = bf16_hi(w[e]);
        s = fmaf(a, a, s);
        s = fmaf(b, b, s);
    }
    return s;
}

// Qwen3 RMSNorm on 8 bf16 values: bf16(gamma * bf16(x * r)).
__device__ __forceinline__ uint4 norm8(uint4 v, uint4 g, float r) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w}, gw[4] = {g.x, g.y, g.z, g.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
        o[e] = pack_bf16(bf16_lo(gw[e]) * rbf(bf16_lo(w[e]) * r), bf16_hi(gw[e]) * rbf(bf16_hi(w[e]) * r));
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// RMSNorm ("A modern architecture: Qwen3", section RMSNorm): mean of squares in fp32, r =
// rsqrt(mean + eps) correctly rounded, cast of x*r to bf16, then times gamma. One warp per row;
// rows up to 32*8*CACHE elements stay in registers, longer rows are re-read for the second pass.
template <int CACHE>
__global__ void rmsnorm_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ g, int rows,
                               int n, long long in_stride, long long in_offset, float eps,
                               __nv_bfloat16* __restrict__ y) {
    pdl_trigger();  // the next kernel only prefetches weights before its own wait
    pdl_wait();
    const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)(row * in_stride + in_offset) * n);
    const uint4* gr = reinterpret_cast<const uint4*>(g);
    uint4* yr = reinterpret_cast<uint4*>(y + (size_t)row * n);
    const int nv = n / 8;
    uint4 cache[CACHE];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < CACHE; ++i) {
        const int v = lane + 32 * i;
        if (v < nv) {
            cache[i] = xr[v];
            ss += sumsq8(cache[i]);
        }
    }
    for (int v = lane + 32 * CACHE; v < nv; v += 32) ss += sumsq8(xr[v]);
    ss = warp_sum(ss);
    const float r = __frsqrt_rn(ss / (float)n + eps);
#pragma unroll
    for (int i = 0; i < CACHE; ++i) {
        const int v = lane + 32 * i;
        if (v < nv) yr[v] = norm8(cache[i], __ldg(gr + v), r);
    }
    for (int v = lane + 32 * CACHE; v < nv; v += 32) yr[v] = norm8(xr[v], __ldg(gr + v), r);
}

// RoPE table row p: cos(fp32(p * w_i)) for i < dh/2, then sin(...), each rounded fp32 -> bf16, with
// w_i = fp32(theta^(-2i/dh)) ("A modern architecture: Qwen3", Rotary position embeddings,
// rope_cos_sin). Built once per context; the transcendental functions run in fp64 and are rounded
// to fp32, so the table holds the correctly rounded fp32 values before the bf16 cast.
__global__ void rope_table_kernel(double theta, int dh, int n_pos, __nv_bfloat16* __restrict__ table) {
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const int half = dh / 2;
    if (idx >= (long long)n_pos * half) return;
    const int p = (int)(idx / half), i = (int)(idx % half);
    const float w = (float)pow(theta, -2.0 * i / dh);
    const float ang = (float)p * w;
    const float c = (float)cos((double)ang), s = (float)sin((double)ang);
    table[(size_t)p * dh + i] = __float2bfloat16_rn(c);
    table[(size_t)p * dh + half + i] = __float2bfloat16_rn(s);
}

// Fused per-head q_norm / k_norm, RoPE and cache append ("A modern architecture: Qwen3", Attention
// with grouped KV heads and Q/K normalization; checklist items on q/k norm before RoPE, V untouched,
// rotate-half pairing). One warp per (token, head) vector of DH values; lane l holds features
// [l*E, l*E+E), so feature i < DH/2 and its rotation partner i + DH/2 sit in lanes l and l^16.
// The rotation is evaluated as bf16(bf16(a*c) + bf16(-b*s)) and bf16(bf16(b*c) + bf16(a*s)).
// F32_SRC: the projection is the sum of the fp32 split-K slices ([splits][B][H*DH], added in order)
// instead of a bf16 qkv buffer; it is rounded to bf16 as the unsplit GEMM stores it.
template <int DH, bool F32_SRC>
__global__ void qknorm_rope_append_kernel(const __nv_bfloat16* __restrict__ qkv, const float* __restrict__ ws, int splits, int B, int T,
                                          int Hq, int Hkv, const __nv_bfloat16* __restrict__ qg,
                                          const __nv_bfloat16* __restrict__ kg, const __nv_bfloat16* __restrict__ table,
                                          const int* __restrict__ len0p, float eps, __nv_bfloat16* __restrict__ q_out,
                                          __nv_bfloat16* __restrict__ kc, __nv_bfloat16* __restrict__ vc, int cap,
                                          const int* __restrict__ meta, int rolling) {
    pdl_wait();
    pdl_trigger();
    constexpr int E = DH / 32;  // 2 or 4 features per lane
    constexpr int HALF = DH / 2;
    const int H = Hq + 2 * Hkv;
    const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (w >= (long long)B * T * H) return;
    const int hh = (int)(w % H);
    const long long m = w / H;
    const int b = (int)(m / T), t = (int)(m % T);
    const int slot = *len0p + t;
    const int pos = meta ? slot_position(slot, meta[0], meta[kSeqMetaHead + b]) : slot;
    const int phys = rolling ? slot % cap : slot;  // cache slot: a rolling buffer wraps

    uint32_t raw[E / 2];
    if constexpr (F32_SRC) {
        const size_t slice = (size_t)B * H * DH;
        const float* src = ws + (size_t)m * H * DH + (size_t)hh * DH + lane * E;
        float acc[E];
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll 4
        for (int sp = 0; sp < splits; ++sp)
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] += src[sp * slice + e];
#pragma unroll
        for (int e = 0; e < E / 2; ++e) raw[e] = pack_bf16(acc[2 * e], acc[2 * e + 1]);
    } else {
        const __nv_bfloat16* src = qkv + (size_t)m * H * DH + (size_t)hh * DH + lane * E;
        if constexpr (E == 4) {
            uint2 v = *reinterpret_cast<const uint2*>(src);
            raw[0] = v.x;
            raw[1] = v.y;
        } else {
            raw[0] = *reinterpret_cast<const uint32_t*>(src);
        }
    }
    if (hh >= Hq + Hkv) {  // V: copied into the cache unchanged
        __nv_bfloat16* dst = vc + (((size_t)b * Hkv + (hh - Hq - Hkv)) * cap + phys) * DH + lane * E;
        if constexpr (E == 4) *reinterpret_cast<uint2*>(dst) = make_uint2(raw[0], raw[1]);
        else *reinterpret_cast<uint32_t*>(dst) = raw[0];
        return;
    }
    float x[E];
#pragma unroll
    for (int e = 0; e < E / 2; ++e) {
        x[2 * e] = bf16_lo(raw[e]);
        x[2 * e + 1] = bf16_hi(raw[e]);
    }
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) ss = fmaf(x[e], x[e], ss);
    ss = warp_sum(ss);
    const float r = __frsqrt_rn(ss / (float)DH + eps);
    const bool is_q = hh < Hq;
    const __nv_bfloat16* gam = (is_q ? qg : kg) + lane * E;
    float y[E];
#pragma unroll
    for (int e = 0; e < E; ++e) y[e] = rbf(bf16f(gam[e]) * rbf(x[e] * r));

    const bool first = lane < 16;
    const int i0 = (lane * E) % HALF;
    const __nv_bfloat16* cs = table + (size_t)pos * DH;
    uint32_t o[E / 2];
#pragma unroll
    for (int e = 0; e < E; e += 2) {
        float res[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float own = y[e + k];
            const float other = __shfl_xor_sync(0xffffffffu, own, 16);
            const float c = bf16f(cs[i0 + e + k]), s = bf16f(cs[HALF + i0 + e + k]);
            res[k] = first ? rbf(rbf(own * c) + rbf(-(other * s))) : rbf(rbf(own * c) + rbf(other * s));
        }
        o[e / 2] = pack_bf16(res[0], res[1]);
    }
    __nv_bfloat16* dst;
    if (is_q) dst = q_out + (((size_t)b * Hq + hh) * T + t) * DH + lane * E;
    else dst = kc + (((size_t)b * Hkv + (hh - Hq)) * cap + phys) * DH + lane * E;
    if constexpr (E == 4) *reinterpret_cast<uint2*>(dst) = make_uint2(o[0], o[1]);
    else *reinterpret_cast<uint32_t*>(dst) = o[0];
}


// x = bf16(x + bf16(acc)) for the decode rows (acc = the sum of the split-K slices, added in order),
// then y = RMSNorm(x) with gain g: the residual add of o_proj / down_proj fused with the RMSNorm that
// follows it (post-attention norm, the next layer's input norm, or the final norm). A row is spread
// over n / FIN_COLS CTAs: each adds its columns, stores x and its partial sum of squares; the last
// CTA of the row (ticket) adds the partials in chunk order and normalises the whole row, so the
// result does not depend on which CTA finishes last. part [M][chunks] and tick [M] are scratch; the
// tickets are zero on entry and left zero.
constexpr int FIN_THREADS = 128, FIN_COLS = FIN_THREADS * 4;
__global__ void __launch_bounds__(FIN_THREADS)
    finalize_residual_rmsnorm_kernel(const float* __restrict__ ws, int splits, long long ldw,
                                     __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ g, int M, int n,
                                     float eps, __nv_bfloat16* __restrict__ y, float* __restrict__ part,
                                     int* __restrict__ tick) {
    pdl_trigger();  // the next kernel only prefetches weights before its own wait
    pdl_wait();
    __shared__ float red[FIN_THREADS / 32];
    __shared__ int last;
    const int row = blockIdx.x, chunk = blockIdx.y, chunks = gridDim.y;
    const int col = chunk * FIN_COLS + threadIdx.x * 4;
    const size_t slice = (size_t)M * ldw;
    float ss = 0.f;
    if (col < n) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const float* wr = ws + (size_t)row * ldw + col;
#pragma unroll 4
        for (int sp = 0; sp < splits; ++sp) {
            const float4 a = *reinterpret_cast<const float4*>(wr + sp * slice);
            acc[0] += a.x, acc[1] += a.y, acc[2] += a.z, acc[3] += a.w;
        }
        uint2* xp = reinterpret_cast<uint2*>(x + (size_t)row * n + col);
        const uint2 xv = *xp;
        const uint32_t xw[2] = {xv.x, xv.y};
        uint32_t o[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            o[e] = pack_bf16(bf16_lo(xw[e]) + rbf(acc[2 * e]), bf16_hi(xw[e]) + rbf(acc[2 * e + 1]));
            const float rl = bf16_lo(o[e]), rh = bf16_hi(o[e]);
            ss = fmaf(rl, rl, ss);
            ss = fmaf(rh, rh, ss);
        }
        *xp = make_uint2(o[0], o[1]);
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < FIN_THREADS / 32; ++w) tot += red[w];
        part[(size_t)row * chunks + chunk] = tot;
        __threadfence();
        last = atomicAdd(&tick[row], 1) == chunks - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    float tot = 0.f;
    for (int c = 0; c < chunks; ++c) tot += part[(size_t)row * chunks + c];  // fixed order
    const float r = __frsqrt_rn(tot / (float)n + eps);
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)row * n);
    const uint4* gr = reinterpret_cast<const uint4*>(g);
    uint4* yr = reinterpret_cast<uint4*>(y + (size_t)row * n);
    for (int v = threadIdx.x; v < n / 8; v += FIN_THREADS) yr[v] = norm8(xr[v], __ldg(gr + v), r);
    if (threadIdx.x == 0) tick[row] = 0;  // ready for the next launch
}

// The same with one 256-thread CTA per row (rows of up to 4096 elements stay in registers); used when
// there are enough rows to fill the GPU without splitting them.
constexpr int FIN_ROW_THREADS = 256;
__global__ void __launch_bounds__(FIN_ROW_THREADS)
    finalize_residual_rmsnorm_row_kernel(const float* __restrict__ ws, int splits, long long ldw,
                                     __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ g, int M, int n,
                                     float eps, __nv_bfloat16* __restrict__ y) {
    pdl_trigger();  // the next kernel only prefetches weights before its own wait
    pdl_wait();
    __shared__ float red[FIN_ROW_THREADS / 32];
    const int row = blockIdx.x;
    constexpr int MAXG = 2;  // 8-element groups per thread: rows up to 256 * 8 * 2 = 4096 elements
    uint4 keep[MAXG];
    float ss = 0.f;
    uint4* xr = reinterpret_cast<uint4*>(x + (size_t)row * n);
    const size_t slice = (size_t)M * ldw;
#pragma unroll
    for (int i = 0; i < MAXG; ++i) {
        const int v = threadIdx.x + FIN_ROW_THREADS * i;
        if (v < n / 8) {
            const uint4 xv = xr[v];
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            const float4* wr = reinterpret_cast<const float4*>(ws + (size_t)row * ldw) + 2 * v;
#pragma unroll 4
            for (int sp = 0; sp < splits; ++sp) {
                const float4 a0 = wr[sp * (slice / 4)], a1 = wr[sp * (slice / 4) + 1];
                acc[0] += a0.x, acc[1] += a0.y, acc[2] += a0.z, acc[3] += a0.w;
                acc[4] += a1.x, acc[5] += a1.y, acc[6] += a1.z, acc[7] += a1.w;
            }
            const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float lo = bf16_lo(xw[e]) + rbf(acc[2 * e]), hi = bf16_hi(xw[e]) + rbf(acc[2 * e + 1]);
                o[e] = pack_bf16(lo, hi);
                const float rl = bf16_lo(o[e]), rh = bf16_hi(o[e]);
                ss = fmaf(rl, rl, ss);
                ss = fmaf(rh, rh, ss);
            }
            keep[i] = make_uint4(o[0], o[1], o[2], o[3]);
            xr[v] = keep[i];
        }
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < FIN_ROW_THREADS / 32; ++w) tot += red[w];
    const float r = __frsqrt_rn(tot / (float)n + eps);
    const uint4* gr = reinterpret_cast<const uint4*>(g);
    uint4* yr = reinterpret_cast<uint4*>(y + (size_t)row * n);
#pragma unroll
    for (int i = 0; i < MAXG; ++i) {
        const int v = threadIdx.x + FIN_ROW_THREADS * i;
        if (v < n / 8) yr[v] = norm8(keep[i], __ldg(gr + v), r);
    }
}

// h = bf16(bf16(silu(bf16(gate))) * bf16(up)) from the split-K slices of the packed gate/up GEMM
// (128-column blocks: gate block j at columns 256j.., up block at 256j+128..).
__global__ void finalize_swiglu_kernel(const float* __restrict__ ws, int splits, long long ldw,
                                       __nv_bfloat16* __restrict__ h, int M, int F) {
    pdl_trigger();  // the next kernel only prefetches weights before its own wait
    pdl_wait();
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // one thread per 4 outputs
    if (idx >= (long long)M * F / 4) return;
    const int row = (int)(idx / (F / 4)), j = (int)(idx % (F / 4)) * 4;
    const size_t slice = (size_t)M * ldw, off = (size_t)row * ldw + (j / 128) * 256 + (j % 128);
    float gg[4] = {0.f, 0.f, 0.f, 0.f}, uu[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int sp = 0; sp < splits; ++sp) {
        const float4 gv = *reinterpret_cast<const float4*>(ws + sp * slice + off);
        const float4 uv = *reinterpret_cast<const float4*>(ws + sp * slice + off + 128);
        gg[0] += gv.x, gg[1] += gv.y, gg[2] += gv.z, gg[3] += gv.w;
        uu[0] += uv.x, uu[1] += uv.y, uu[2] += uv.z, uu[3] += uv.w;
    }
    float o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float g0 = rbf(gg[e]);
        o[e] = rbf(__fdividef(g0, 1.0f + __expf(-g0))) * rbf(uu[e]);
    }
    *reinterpret_cast<uint2*>(h + (size_t)row * F + j) = make_uint2(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]));
}

__global__ void set_len_kernel(int* len, int value) {
    pdl_wait();
    pdl_trigger();
    *len = value;
}
__global__ void add_len_kernel(int* len, int delta) {
    pdl_wait();
    pdl_trigger();
    *len += delta;
}

// Greedy next token ("A modern architecture: Qwen3", generation: argmax of the last row's logits):
// the largest logit, the lowest index on ties, a NaN counting as the largest (torch.argmax's rule).
// A row is split over P CTAs (grid P x B) so that a decode batch of a few rows still streams its
// logits with most SMs: each CTA reduces a segment to one candidate, and the last CTA of the row to
// finish (a ticket per row) picks the best candidate. The comparison is a total order, so the result
// does not depend on which CTA finishes last. With stop_id >= 0 a finished row emits stop_id, and a
// row that emits it is finished; `alive` counts the rows still running after this step.
constexpr int GREEDY_THREADS = 512, GREEDY_UNROLL = 4, GREEDY_MAX_PARTS = 32, GREEDY_TICKETS_PAD = 64;
__device__ __forceinline__ bool greedy_better(float v, int i, float bv, int bi) {
    const bool nv = v != v, nb = bv != bv;
    if (nv != nb) return nv;
    if (nv) return i < bi;
    return v > bv || (v == bv && i < bi);
}
__device__ __forceinline__ void greedy_warp_best(float& bv, int& bi) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (greedy_better(ov, oi, bv, bi)) {
            bv = ov;
            bi = oi;
        }
    }
}
// work: [GREEDY_TICKETS_PAD rounded up to B] ticket ints (zero on entry, left zero), then [B][P] candidates
// (value bits, index); unused when P == 1.
__global__ void __launch_bounds__(GREEDY_THREADS)
    greedy_kernel(const float* __restrict__ logits, long long ld, int V, int stop_id, int* __restrict__ done,
                  int* __restrict__ next, int* __restrict__ out, long long out_ld, int out_col, int* __restrict__ alive,
                  int* __restrict__ work, int tickets) {
    pdl_wait();
    pdl_trigger();
    const int p = blockIdx.x, P = gridDim.x, b = blockIdx.y;
    const float* row = logits + (size_t)b * ld;
    const int seg = ((V + P - 1) / P + 3) / 4 * 4;  // a multiple of 4 floats: every float4 load stays aligned
    const int lo = p * seg, hi = min(V, lo + seg);
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    // GREEDY_UNROLL independent 16-byte loads in flight per thread
    for (int base = lo + threadIdx.x * 4; base < hi; base += GREEDY_THREADS * 4 * GREEDY_UNROLL) {
        float4 v[GREEDY_UNROLL];
#pragma unroll
        for (int u = 0; u < GREEDY_UNROLL; ++u) {
            const int i = base + u * GREEDY_THREADS * 4;
            v[u] = i < hi ? __ldg(reinterpret_cast<const float4*>(row + i)) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
#pragma unroll
        for (int u = 0; u < GREEDY_UNROLL; ++u) {
            const int i = base + u * GREEDY_THREADS * 4;
            const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (i + k < hi && greedy_better(e[k], i + k, bv, bi)) {
                    bv = e[k];
                    bi = i + k;
                }
        }
    }
    greedy_warp_best(bv, bi);
    __shared__ float sv[GREEDY_THREADS / 32];
    __shared__ int si[GREEDY_THREADS / 32];
    __shared__ int last;
    if ((threadIdx.x & 31) == 0) {
        sv[threadIdx.x >> 5] = bv;
        si[threadIdx.x >> 5] = bi;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        bv = threadIdx.x < GREEDY_THREADS / 32 ? sv[threadIdx.x] : -INFINITY;
        bi = threadIdx.x < GREEDY_THREADS / 32 ? si[threadIdx.x] : 0x7fffffff;
        greedy_warp_best(bv, bi);
    }
    if (P > 1) {
        int* tick = work + b;
        int2* cand = reinterpret_cast<int2*>(work + tickets) + (size_t)b * P;
        if (threadIdx.x == 0) {
            cand[p] = make_int2(__float_as_int(bv), bi);
            __threadfence();
            last = atomicAdd(tick, 1) == P - 1;
        }
        __syncthreads();
        if (!last) return;
        if (threadIdx.x >= 32) return;
        __threadfence();
        const int2 c = threadIdx.x < P ? __ldcg(cand + threadIdx.x) : make_int2(__float_as_int(-INFINITY), 0x7fffffff);
        bv = __int_as_float(c.x);
        bi = c.y;
        greedy_warp_best(bv, bi);
        if (threadIdx.x == 0) *tick = 0;  // ready for the next launch
    }
    if (threadIdx.x == 0) {
        if (bi >= V) bi = 0;  // every logit was -inf: the first index, as argmax returns
        int tok = bi;
        if (stop_id >= 0 && done) {
            const int was = done[b];
            if (was) tok = stop_id;
            const int fin = was || tok == stop_id;
            done[b] = fin;
            if (alive && !fin) atomicAdd(alive, 1);
        }
        if (next) next[b] = tok;
        if (out) out[(size_t)b * out_ld + out_col] = tok;
    }
}

// Sequence layout update: writes n ints carried in the launch itself (no host buffer to keep alive,
// stream-ordered like every other launch).
struct SeqChunk {
    int v[kSeqChunk];
};
__global__ void set_seq_kernel(int* __restrict__ dst, SeqChunk c, int n) {
    pdl_wait();
    pdl_trigger();
    for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = c.v[i];
}

// Shared prefix: copy cache slots [s0, s1) of sequence 0 into sequences 1..nb-1, every layer and kv
// head, K and V (the part of a shared prefix that does not fill a whole 128-slot tile).
__global__ void copy_prefix_slots_kernel(__nv_bfloat16* __restrict__ kc, __nv_bfloat16* __restrict__ vc,
                                         size_t layer_elems, int Hkv, int cap, int dh, int s0, int s1) {
    const int j = blockIdx.x, bdst = blockIdx.y + 1, l = blockIdx.z;
    const size_t src = (size_t)l * layer_elems + ((size_t)j * cap + s0) * dh;
    const size_t dst = (size_t)l * layer_elems + (((size_t)bdst * Hkv + j) * cap + s0) * dh;
    const int n = (s1 - s0) * dh / 8;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        reinterpret_cast<uint4*>(kc + dst)[i] = reinterpret_cast<const uint4*>(kc + src)[i];
        reinterpret_cast<uint4*>(vc + dst)[i] = reinterpret_cast<const uint4*>(vc + src)[i];
    }
}

}  // namespace

cudaError_t embed_launch(const __nv_bfloat16* E, int V, int d, const int32_t* ids, int M, __nv_bfloat16* out, int* err,
                         cudaStream_t st) {
    if (M <= 0) return cudaSuccess;
    const int threads = 256, rows_per_block = threads / 32;
    return launch_pdl(embed_kernel, dim3((M + rows_per_block - 1) / rows_per_block), dim3(threads), 0, st, E, V, d, ids,
                      M, out, err);
}

cudaError_t rmsnorm_launch(const __nv_bfloat16* x, const __nv_bfloat16* g, int rows, int n, long long in_stride,
                           long long in_offset, float eps, __nv_bfloat16* y, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    const int threads = 128, rpb = threads / 32;
    const int blocks = (rows + rpb - 1) / rpb;
    if (n <= 32 * 8 * 4)
        return launch_pdl(rmsnorm_kernel<4>, dim3(blocks), dim3(threads), 0, st, x, g, rows, n, in_stride, in_offset, eps,
                          y);
    return launch_pdl(rmsnorm_kernel<16>, dim3(blocks), dim3(threads), 0, st, x, g, rows, n, in_stride, in_offset, eps, y);
}

cudaError_t rope_table_launch(float theta, int dh, int n_pos, __nv_bfloat16* table, cudaStream_t st) {
    const long long n = (long long)n_pos * (dh / 2);
    if (n <= 0) return cudaSuccess;
    rope_table_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>((double)theta, dh, n_pos, table);
    return cudaGetLastError();
}

cudaError_t pack_gate_up_launch(const __nv_bfloat16* gate, const __nv_bfloat16* up, int F, int d, __nv_bfloat16* out,
                                cudaStream_t st) {
    // out rows [256j, 256j+128) = gate rows [128j, 128j+128); [256j+128, 256j+256) = up rows.
    const size_t block_bytes = (size_t)128 * d * 2;
    cudaError_t e = cudaMemcpy2DAsync(out, 2 * block_bytes, gate, block_bytes, block_bytes, F / 128,
                                      cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return e;
    return cudaMemcpy2DAsync(reinterpret_cast<char*>(out) + block_bytes, 2 * block_bytes, up, block_bytes, block_bytes,
                             F / 128, cudaMemcpyDeviceToDevice, st);
}

cudaError_t qknorm_rope_append_launch(const __nv_bfloat16* qkv, int B, int T, int Hq, int Hkv, int dh,
                                      const __nv_bfloat16* qg, const __nv_bfloat16* kg, const __nv_bfloat16* table,
                                      const int* len0, float eps, __nv_bfloat16* q_out, __nv_bfloat16* kc,
                                      __nv_bfloat16* vc, int cap, cudaStream_t st) {
    const long long warps = (long long)B * T * (Hq + 2 * Hkv);
    if (warps <= 0) return cudaSuccess;
    const int threads = 256, wpb = threads / 32;
    const unsigned blocks = (unsigned)((warps + wpb - 1) / wpb);
    const float* nows = nullptr;
    const int* nometa = nullptr;
    if (dh == 128)
        return launch_pdl(qknorm_rope_append_kernel<128, false>, dim3(blocks), dim3(threads), 0, st, qkv, nows, 1, B, T, Hq,
                          Hkv, qg, kg, table, len0, eps, q_out, kc, vc, cap, nometa, 0);
    if (dh == 64)
        return launch_pdl(qknorm_rope_append_kernel<64, false>, dim3(blocks), dim3(threads), 0, st, qkv, nows, 1, B, T, Hq,
                          Hkv, qg, kg, table, len0, eps, q_out, kc, vc, cap, nometa, 0);
    return cudaErrorInvalidValue;
}

cudaError_t set_len_launch(int* len, int value, cudaStream_t st) {
    return launch_pdl(set_len_kernel, dim3(1), dim3(1), 0, st, len, value);
}

cudaError_t add_len_launch(int* len, int delta, cudaStream_t st) {
    return launch_pdl(add_len_kernel, dim3(1), dim3(1), 0, st, len, delta);
}

int finalize_norm_chunks(int n) { return (n + FIN_COLS - 1) / FIN_COLS; }

cudaError_t finalize_residual_rmsnorm_launch(const float* ws, int splits, long long ldw, __nv_bfloat16* x,
                                             const __nv_bfloat16* g, int M, int n, float eps, __nv_bfloat16* y,
                                             float* part, int* tick, cudaStream_t st) {
    if (M <= 0) return cudaSuccess;
    if (n % 8 || ldw % 4 || !part || !tick) return cudaErrorInvalidValue;
    if (M >= 32 && n <= 4096)
        return launch_pdl(finalize_residual_rmsnorm_row_kernel, dim3(M), dim3(FIN_ROW_THREADS), 0, st, ws, splits, ldw, x,
                          g, M, n, eps, y);
    return launch_pdl(finalize_residual_rmsnorm_kernel, dim3(M, finalize_norm_chunks(n)), dim3(FIN_THREADS), 0, st, ws,
                      splits, ldw, x, g, M, n, eps, y, part, tick);
}

cudaError_t finalize_swiglu_launch(const float* ws, int splits, long long ldw, __nv_bfloat16* h, int M, int F,
                                   cudaStream_t st) {
    if (M <= 0) return cudaSuccess;
    const long long n = (long long)M * F / 4;
    return launch_pdl(finalize_swiglu_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, ws, splits, ldw, h, M,
                      F);
}

cudaError_t qknorm_rope_append_f32_launch(const float* ws, int splits, int B, int Hq, int Hkv, int dh,
                                          const __nv_bfloat16* qg, const __nv_bfloat16* kg, const __nv_bfloat16* table,
                                          const int* len0, float eps, __nv_bfloat16* q_out, __nv_bfloat16* kc,
                                          __nv_bfloat16* vc, int cap, const int* meta, int rolling, cudaStream_t st) {
    const long long warps = (long long)B * (Hq + 2 * Hkv);
    if (warps <= 0) return cudaSuccess;
    const int threads = 256, wpb = threads / 32;
    const unsigned blocks = (unsigned)((warps + wpb - 1) / wpb);
    const __nv_bfloat16* noq = nullptr;
    if (dh == 128)
        return launch_pdl(qknorm_rope_append_kernel<128, true>, dim3(blocks), dim3(threads), 0, st, noq, ws, splits, B, 1,
                          Hq, Hkv, qg, kg, table, len0, eps, q_out, kc, vc, cap, meta, rolling);
    if (dh == 64)
        return launch_pdl(qknorm_rope_append_kernel<64, true>, dim3(blocks), dim3(threads), 0, st, noq, ws, splits, B, 1,
                          Hq, Hkv, qg, kg, table, len0, eps, q_out, kc, vc, cap, meta, rolling);
    return cudaErrorInvalidValue;
}

int greedy_parts(int B, int V) {
    const int per_cta = GREEDY_THREADS * 4 * GREEDY_UNROLL;  // floats one CTA pass covers
    const int max_p = (V + per_cta - 1) / per_cta;
    const int want = (2 * device_sm_count() + B - 1) / std::max(B, 1);
    return std::max(1, std::min(std::min(max_p, want), GREEDY_MAX_PARTS));
}

size_t greedy_workspace_ints(int B) {
    const int tickets = (std::max(B, 1) + GREEDY_TICKETS_PAD - 1) / GREEDY_TICKETS_PAD * GREEDY_TICKETS_PAD;
    return (size_t)tickets + (size_t)std::max(B, 1) * GREEDY_MAX_PARTS * 2;
}

cudaError_t greedy_launch(const float* logits, long long ld, int B, int V, int stop_id, int* done, int* next, int* out,
                          long long out_ld, int out_col, int* alive, int* work, cudaStream_t st) {
    if (B <= 0) return cudaSuccess;
    if (V < 1 || V % 4 || ld % 4) return cudaErrorInvalidValue;
    const int P = work ? greedy_parts(B, V) : 1;
    const int tickets = (B + GREEDY_TICKETS_PAD - 1) / GREEDY_TICKETS_PAD * GREEDY_TICKETS_PAD;
    return launch_pdl(greedy_kernel, dim3(P, B), dim3(GREEDY_THREADS), 0, st, logits, ld, V, stop_id, done, next, out,
                      out_ld, out_col, alive, work, tickets);
}

cudaError_t set_seq_launch(int* dst, const int* vals, int n, cudaStream_t st) {
    for (int i = 0; i < n; i += kSeqChunk) {
        SeqChunk c;
        const int k = std::min(kSeqChunk, n - i);
        for (int j = 0; j < k; ++j) c.v[j] = vals[i + j];
        cudaError_t e = launch_pdl(set_seq_kernel, dim3(1), dim3(256), 0, st, dst + i, c, k);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t copy_prefix_slots_launch(__nv_bfloat16* kc, __nv_bfloat16* vc, size_t layer_elems, int L, int nb, int Hkv,
                                     int cap, int dh, int s0, int s1, cudaStream_t st) {
    if (nb <= 1 || s1 <= s0) return cudaSuccess;
    copy_prefix_slots_kernel<<<dim3(Hkv, nb - 1, L), 256, 0, st>>>(kc, vc, layer_elems, Hkv, cap, dh, s0, s1);
    return cudaGetLastError();
}

}  // namespace q3
