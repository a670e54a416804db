// Qwen3 decoder oracle: plain single-threaded CPU implementation.
//
// TEST INFRASTRUCTURE ONLY (see qwen3_oracle.h). Nothing here is blocked, fused or reordered
// beyond what the pages' definitions state; each loop is the definition written out.
//
// Sources ("A modern architecture: Qwen3" = inference.shantanugoel.com/17-qwen3; "checklist" =
// the Qwen3 block checklist page; "modern architectures lesson" = transformer-architectures-06):
//   RMSNorm             - A modern architecture: Qwen3, section RMSNorm (formula, worked example
//                         [3,4] -> [0.8485, 1.1314], parity details 1-2); checklist, RMSNorm item.
//   RoPE                - same page, section Rotary position embeddings (R(phi), omega_i =
//                         theta^(-2i/d), split-half pairing, rope_cos_sin / apply_rope).
//   q/k norm, GQA       - same page, section Attention with grouped KV heads and Q/K normalization;
//                         checklist items on q_norm/k_norm and GQA; modern architectures lesson,
//                         section 3 (query head h reads kv head floor(h/g)).
//   SwiGLU              - same page, section SwiGLU (SiLU(2) = 1.7616 worked example).
//   Block / model       - same page, section The whole model (pre-norm block, final norm, tied head).
//
// Parity status: every function below is pinned by a test in tests/test_oracle_*.py against a
// value the pages print, a closed form, an invariant, or an independent library routine, except
// oracle_forward as a whole, which is pinned only through its pinned parts plus invariants
// (cached == uncached, causal prefix, batch independence) and an fp64 library re-statement.
// The masked forms (oracle_attention_masked_gqa_row_f64, oracle_layer_out_masked,
// oracle_forward_masked) are pinned by reduction to the equal-length forward pass and by the pairs
// of routes the pages say must agree: a padded row equals the row alone, a shared prefix equals the
// concatenated prompt, a banded mask equals a rolling buffer (tests/test_oracle_generation.py).

#include "qwen3_oracle.h"

#include <cmath>
#include <cstring>
#include <vector>

namespace {

inline float f32_of(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

// float -> bf16, round to nearest even (the conversion PyTorch's .to(torch.bfloat16) performs).
inline uint16_t bf16_of(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)(((u >> 16) & 0x8000u) | 0x7fc0u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

// double -> bf16 with a single rounding. Rounding to float first is exact unless the float lands
// on a bf16 midpoint that the true value does not sit on; that case is resolved from the sign of
// the float's rounding error.
inline uint16_t bf16_of_d(double x) {
    if (std::isnan(x)) return 0x7fc0;
    float f = (float)x;
    uint32_t u;
    std::memcpy(&u, &f, 4);
    if ((u & 0xffffu) == 0x8000u && (double)f != x && std::isfinite(f)) {
        bool above = std::fabs(x) > std::fabs((double)f);
        return (uint16_t)(above ? ((u + 0x10000u) >> 16) : (u >> 16));
    }
    return bf16_of(f);
}

struct Dims {
    int L, d, hq, hkv, dh, F, V, tie, g;
    double theta, eps;
    explicit Dims(const oracle_config* c)
        : L(c->n_layers), d(c->hidden), hq(c->n_q_heads), hkv(c->n_kv_heads), dh(c->head_dim),
          F(c->intermediate), V(c->vocab), tie(c->tie_embeddings), g(c->n_q_heads / c->n_kv_heads),
          theta(c->rope_theta), eps(c->rms_eps) {}
};

}  // namespace

extern "C" {

uint16_t oracle_bf16_from_f32(float x) { return bf16_of(x); }
uint16_t oracle_bf16_from_f64(double x) { return bf16_of_d(x); }
float oracle_f32_from_bf16(uint16_t h) { return f32_of(h); }

// RMSNorm, fp32 stage: x32 * rsqrt(mean(x32^2) + eps). The mean of the squares is the exact mean
// rounded to fp32; eps is added in fp32; rsqrt is the correctly rounded fp32 value.
void oracle_rmsnorm_core_f32(const float* x, int n, double eps, float* y) {
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += (double)x[i] * (double)x[i];
    float mean = (float)(s / n);
    float var = mean + (float)eps;
    float r = (float)(1.0 / std::sqrt((double)var));
    for (int i = 0; i < n; ++i) y[i] = x[i] * r;
}

// Qwen3 RMSNorm on bf16 rows: normalise in fp32, cast to bf16, then multiply by gamma in bf16.
void oracle_rmsnorm(const uint16_t* x, const uint16_t* gamma, int64_t rows, int n, double eps, uint16_t* y) {
    std::vector<float> xf(n), yf(n);
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* xr = x + r * n;
        for (int i = 0; i < n; ++i) xf[i] = f32_of(xr[i]);
        oracle_rmsnorm_core_f32(xf.data(), n, eps, yf.data());
        for (int i = 0; i < n; ++i) {
#ifdef ORACLE_PLANT_GAMMA_BEFORE_CAST
            y[r * n + i] = bf16_of(f32_of(gamma[i]) * yf[i]);
#else
            float cast = f32_of(bf16_of(yf[i]));
            y[r * n + i] = bf16_of(f32_of(gamma[i]) * cast);
#endif
        }
    }
}

// y[m][n] = bf16( sum_k a[m][k] * w[n][k] ), nn.Linear without bias.
void oracle_linear(const uint16_t* a, const uint16_t* w, int64_t M, int64_t N, int64_t K, uint16_t* y) {
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0;
            const uint16_t* ar = a + m * K;
            const uint16_t* wr = w + n * K;
#ifdef ORACLE_PLANT_LINEAR_DROP_LAST_K
            for (int64_t k = 0; k + 1 < K; ++k) s += (double)f32_of(ar[k]) * (double)f32_of(wr[k]);
#else
            for (int64_t k = 0; k < K; ++k) s += (double)f32_of(ar[k]) * (double)f32_of(wr[k]);
#endif
            y[m * N + n] = bf16_of_d(s);
        }
}

void oracle_linear_f32out(const uint16_t* a, const uint16_t* w, int64_t M, int64_t N, int64_t K, float* y) {
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0;
            const uint16_t* ar = a + m * K;
            const uint16_t* wr = w + n * K;
            for (int64_t k = 0; k < K; ++k) s += (double)f32_of(ar[k]) * (double)f32_of(wr[k]);
            y[m * N + n] = (float)s;
        }
}

// Residual add on bf16 tensors: out = bf16(x + y) ("A modern architecture: Qwen3", The whole model:
// x = x + self_attn(...), x + mlp(...)).
void oracle_residual_add(const uint16_t* x, const uint16_t* y, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_of(f32_of(x[i]) + f32_of(y[i]));
}

// SiLU(z) = z * sigmoid(z).
double oracle_silu(double z) {
#ifdef ORACLE_PLANT_SILU_SIGN
    return z / (1.0 + std::exp(z));
#else
    return z / (1.0 + std::exp(-z));
#endif
}

// SwiGLU hidden activation: silu(gate) * up, each op rounded to bf16.
void oracle_swiglu(const uint16_t* g, const uint16_t* u, int64_t n, uint16_t* a) {
    for (int64_t i = 0; i < n; ++i) {
        float s = f32_of(bf16_of_d(oracle_silu((double)f32_of(g[i]))));
        a[i] = bf16_of(s * f32_of(u[i]));
    }
}

// omega_i = theta^(-2i/d), i = 0 .. d/2-1, correctly rounded to fp32.
void oracle_rope_inv_freq(double theta, int dim, float* inv) {
    for (int i = 0; i < dim / 2; ++i) inv[i] = (float)std::pow(theta, -2.0 * i / dim);
}

// cos/sin of the fp32 angle pos * omega_i, computed in fp32 and cast to bf16.
void oracle_rope_cos_sin(int64_t pos, const float* inv, int half, uint16_t* cos_out, uint16_t* sin_out) {
    float p = (float)pos;
    for (int i = 0; i < half; ++i) {
        float ang = p * inv[i];
        cos_out[i] = bf16_of((float)std::cos((double)ang));
        sin_out[i] = bf16_of((float)std::sin((double)ang));
    }
}

// x*cos + rotate_half(x)*sin with rotate_half(x) = cat(-x2, x1): feature i pairs with i + dim/2.
// Each product and the sum are bf16 ops.
void oracle_rope_apply(uint16_t* x, int dim, const uint16_t* cos_t, const uint16_t* sin_t) {
    int h = dim / 2;
    for (int i = 0; i < h; ++i) {
#ifdef ORACLE_PLANT_ROPE_ADJACENT
        int ia = 2 * i, ib = 2 * i + 1;
#else
        int ia = i, ib = i + h;
#endif
        float a = f32_of(x[ia]), b = f32_of(x[ib]);
        float c = f32_of(cos_t[i]), s = f32_of(sin_t[i]);
#ifdef ORACLE_PLANT_ROPE_SIGN
        s = -s;
#endif
        float ac = f32_of(bf16_of(a * c)), nbs = f32_of(bf16_of(-(b * s)));
        float bc = f32_of(bf16_of(b * c)), as = f32_of(bf16_of(a * s));
        x[ia] = bf16_of(ac + nbs);
        x[ib] = bf16_of(bc + as);
    }
}

// fp64 rotation of each pair (x_i, x_{i+d/2}) by angle pos * omega_i: the R(phi) of the pages.
void oracle_rope_rotate_f64(const double* x, int dim, double pos, const double* omega, double* y) {
    int h = dim / 2;
    for (int i = 0; i < h; ++i) {
        double ang = pos * omega[i], c = std::cos(ang), s = std::sin(ang);
        double a = x[i], b = x[i + h];
        y[i] = a * c - b * s;
        y[i + h] = a * s + b * c;
    }
}

// softmax(q . k_s * scale) weighted sum of v_s over the n given keys.
void oracle_attention_row_f64(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t n,
                              int dim, int64_t kv_stride, double scale, double* out) {
    std::vector<double> sc((size_t)n);
    double m = -INFINITY;
    for (int64_t s = 0; s < n; ++s) {
        double dot = 0.0;
        for (int i = 0; i < dim; ++i) dot += (double)f32_of(q[i]) * (double)f32_of(k[s * kv_stride + i]);
        sc[s] = dot * scale;
        if (sc[s] > m) m = sc[s];
    }
    double den = 0.0;
    for (int64_t s = 0; s < n; ++s) {
        sc[s] = std::exp(sc[s] - m);
        den += sc[s];
    }
    for (int i = 0; i < dim; ++i) {
        double acc = 0.0;
        for (int64_t s = 0; s < n; ++s) acc += sc[s] * (double)f32_of(v[s * kv_stride + i]);
        out[i] = acc / den;
    }
}

// All query heads of one row against keys 0..n-1 of a cache set [Hkv][cap][dh]. Grouped-query
// attention: query head h reads kv head floor(h / g), g = Hq / Hkv (repeat_interleave order).
// Scale is head_dim^-0.5.
void oracle_attention_gqa_row_f64(const uint16_t* q, const uint16_t* kc, const uint16_t* vc, int64_t n,
                                  int hq, int hkv, int dim, int64_t cap, double* out) {
    int g = hq / hkv;
#ifdef ORACLE_PLANT_SCALE_BY_DIM
    double scale = 1.0 / dim;
#else
    double scale = 1.0 / std::sqrt((double)dim);
#endif
    for (int h = 0; h < hq; ++h) {
#ifdef ORACLE_PLANT_GQA_MODULO
        int j = h % hkv;
#else
        int j = h / g;
#endif
        int64_t base = (int64_t)j * cap * dim;
        oracle_attention_row_f64(q + (int64_t)h * dim, kc + base, vc + base, n, dim, dim, scale,
                                 out + (int64_t)h * dim);
    }
}

// Parameter count by part, from the shapes this oracle uses.
void oracle_param_count(const oracle_config* c, int64_t parts[6]) {
    Dims D(c);
    int64_t L = D.L, d = D.d, qw = (int64_t)D.hq * D.dh, kvw = (int64_t)D.hkv * D.dh;
    parts[0] = (int64_t)D.V * d;
    parts[1] = L * (d * qw + 2 * d * kvw + qw * d);
    parts[2] = L * 2 * (int64_t)D.dh;
    parts[3] = L * 3 * d * (int64_t)D.F;
    parts[4] = L * 2 * d + d;
    parts[5] = D.tie ? 0 : (int64_t)D.V * d;
}

// a2-a4: input RMSNorm, separate q/k/v projections, per-head q_norm / k_norm, RoPE on q and k.
void oracle_layer_qkv(const oracle_config* c, const oracle_weights* w, int layer, const uint16_t* xin,
                      const int32_t* pos, int64_t n, uint16_t* q, uint16_t* k, uint16_t* v) {
    Dims D(c);
    int64_t qw = (int64_t)D.hq * D.dh, kvw = (int64_t)D.hkv * D.dh;
    std::vector<uint16_t> xn((size_t)(n * D.d)), tmp((size_t)D.dh);
    oracle_rmsnorm(xin, w->in_norm[layer], n, D.d, D.eps, xn.data());
    oracle_linear(xn.data(), w->q_proj[layer], n, qw, D.d, q);
    oracle_linear(xn.data(), w->k_proj[layer], n, kvw, D.d, k);
    oracle_linear(xn.data(), w->v_proj[layer], n, kvw, D.d, v);
    std::vector<float> inv((size_t)D.dh / 2);
    std::vector<uint16_t> cs((size_t)D.dh / 2), sn((size_t)D.dh / 2);
    oracle_rope_inv_freq(D.theta, D.dh, inv.data());
    for (int64_t r = 0; r < n; ++r) {
        oracle_rope_cos_sin(pos[r], inv.data(), D.dh / 2, cs.data(), sn.data());
        for (int h = 0; h < D.hq; ++h) {
            uint16_t* qh = q + r * qw + (int64_t)h * D.dh;
#ifndef ORACLE_PLANT_NO_QNORM
            oracle_rmsnorm(qh, w->q_norm[layer], 1, D.dh, D.eps, tmp.data());
            std::memcpy(qh, tmp.data(), (size_t)D.dh * 2);
#endif
            oracle_rope_apply(qh, D.dh, cs.data(), sn.data());
        }
        for (int h = 0; h < D.hkv; ++h) {
            uint16_t* kh = k + r * kvw + (int64_t)h * D.dh;
            oracle_rmsnorm(kh, w->k_norm[layer], 1, D.dh, D.eps, tmp.data());
            std::memcpy(kh, tmp.data(), (size_t)D.dh * 2);
            oracle_rope_apply(kh, D.dh, cs.data(), sn.data());
        }
    }
}

// a6-a9 for n rows, given their bf16 attention outputs att [n][Hq*dh]: o_proj + residual,
// post-attention RMSNorm, SwiGLU MLP + residual.
static void layer_tail(const oracle_config* c, const oracle_weights* w, int layer, const uint16_t* xin,
                       const uint16_t* att, int64_t n, uint16_t* xout) {
    Dims D(c);
    int64_t qw = (int64_t)D.hq * D.dh;
    std::vector<uint16_t> o((size_t)(n * D.d)), x1((size_t)(n * D.d)), xn((size_t)(n * D.d)),
        gt((size_t)(n * D.F)), up((size_t)(n * D.F)), a((size_t)(n * D.F)), dn((size_t)(n * D.d));
    oracle_linear(att, w->o_proj[layer], n, D.d, qw, o.data());
#ifdef ORACLE_PLANT_DROP_ATTN_RESIDUAL
    for (int64_t i = 0; i < n * D.d; ++i) x1[i] = o[i];
#else
    oracle_residual_add(xin, o.data(), n * D.d, x1.data());
#endif
    oracle_rmsnorm(x1.data(), w->post_norm[layer], n, D.d, D.eps, xn.data());
    oracle_linear(xn.data(), w->gate_proj[layer], n, D.F, D.d, gt.data());
    oracle_linear(xn.data(), w->up_proj[layer], n, D.F, D.d, up.data());
    oracle_swiglu(gt.data(), up.data(), n * D.F, a.data());
    oracle_linear(a.data(), w->down_proj[layer], n, D.d, D.F, dn.data());
    oracle_residual_add(x1.data(), dn.data(), n * D.d, xout);
}

// a5-a9: causal GQA attention over the cache, o_proj + residual, post-attention RMSNorm,
// SwiGLU MLP + residual.
void oracle_layer_out(const oracle_config* c, const oracle_weights* w, int layer, const uint16_t* xin,
                      const uint16_t* q, const int32_t* pos, int64_t n, const uint16_t* kc,
                      const uint16_t* vc, const int32_t* kvset, int64_t cap, uint16_t* xout) {
    Dims D(c);
    int64_t qw = (int64_t)D.hq * D.dh;
    std::vector<uint16_t> att((size_t)(n * qw));
    std::vector<double> orow((size_t)qw);
    for (int64_t r = 0; r < n; ++r) {
        int64_t set_base = (int64_t)kvset[r] * D.hkv * cap * D.dh;
        oracle_attention_gqa_row_f64(q + r * qw, kc + set_base, vc + set_base, (int64_t)pos[r] + 1,
                                     D.hq, D.hkv, D.dh, cap, orow.data());
        for (int64_t i = 0; i < qw; ++i) att[r * qw + i] = bf16_of_d(orow[i]);
    }
    layer_tail(c, w, layer, xin, att.data(), n, xout);
}

// Masked attention (the pages' boolean attention mask, True = may attend): the keys a row's mask
// admits are gathered in slot order from one cache set kc/vc [Hkv][cap][dh] and handed to the
// plain row attention. A row that admits no key has no defined output (softmax over nothing);
// the function returns -3 for it.
int oracle_attention_masked_gqa_row_f64(const uint16_t* q, const uint16_t* kc, const uint16_t* vc,
                                        int64_t cap, const uint8_t* mask, int hq, int hkv, int dim,
                                        double* out) {
    std::vector<int64_t> keep;
    for (int64_t s = 0; s < cap; ++s) {
#ifdef ORACLE_PLANT_MASK_CAUSAL_ONLY
        // planted mistake: every slot up to the last admitted one, masked keys inside included
        bool later = false;
        for (int64_t u = s; u < cap; ++u) later = later || mask[u];
        if (later) keep.push_back(s);
#else
        if (mask[s]) keep.push_back(s);
#endif
    }
    if (keep.empty()) return -3;
    int64_t n = (int64_t)keep.size();
    std::vector<uint16_t> kg((size_t)(hkv * n * dim)), vg((size_t)(hkv * n * dim));
    for (int j = 0; j < hkv; ++j)
        for (int64_t i = 0; i < n; ++i) {
            std::memcpy(&kg[(size_t)((j * n + i) * dim)], kc + ((int64_t)j * cap + keep[i]) * dim, (size_t)dim * 2);
            std::memcpy(&vg[(size_t)((j * n + i) * dim)], vc + ((int64_t)j * cap + keep[i]) * dim, (size_t)dim * 2);
        }
    oracle_attention_gqa_row_f64(q, kg.data(), vg.data(), n, hq, hkv, dim, n, out);
    return 0;
}

// a5-a9 with an explicit mask per row: row r reads the slots of kv set kvset[r] that
// mask[r][0..cap) admits.
int oracle_layer_out_masked(const oracle_config* c, const oracle_weights* w, int layer, const uint16_t* xin,
                            const uint16_t* q, int64_t n, const uint16_t* kc, const uint16_t* vc,
                            const int32_t* kvset, int64_t cap, const uint8_t* mask, uint16_t* xout) {
    Dims D(c);
    int64_t qw = (int64_t)D.hq * D.dh;
    std::vector<uint16_t> att((size_t)(n * qw));
    std::vector<double> orow((size_t)qw);
    for (int64_t r = 0; r < n; ++r) {
        int64_t set_base = (int64_t)kvset[r] * D.hkv * cap * D.dh;
        int rc = oracle_attention_masked_gqa_row_f64(q + r * qw, kc + set_base, vc + set_base, cap, mask + r * cap,
                                                     D.hq, D.hkv, D.dh, orow.data());
        if (rc != 0) return rc;
        for (int64_t i = 0; i < qw; ++i) att[r * qw + i] = bf16_of_d(orow[i]);
    }
    layer_tail(c, w, layer, xin, att.data(), n, xout);
    return 0;
}

// Final RMSNorm, then hidden @ W^T with W = lm_head, or the embedding matrix when tied.
void oracle_head(const oracle_config* c, const oracle_weights* w, const uint16_t* x, int64_t n, float* logits) {
    Dims D(c);
    std::vector<uint16_t> hn((size_t)(n * D.d));
    oracle_rmsnorm(x, w->final_norm, n, D.d, D.eps, hn.data());
    const uint16_t* W = D.tie ? w->embed : w->lm_head;
    oracle_linear_f32out(hn.data(), W, n, D.V, D.d, logits);
}

int oracle_forward(const oracle_config* c, const oracle_weights* w, uint16_t* kc, uint16_t* vc,
                   int B, int64_t cap, int64_t len0, const int32_t* ids, int T, int all_rows,
                   float* logits, int tap_layer, uint16_t* tap_in, uint16_t* tap_out) {
    Dims D(c);
    if (len0 + T > cap) return -2;
    int64_t M = (int64_t)B * T;
    int64_t qw = (int64_t)D.hq * D.dh, kvw = (int64_t)D.hkv * D.dh;
    std::vector<uint16_t> x((size_t)(M * D.d)), y((size_t)(M * D.d)), q((size_t)(M * qw)),
        k((size_t)(M * kvw)), v((size_t)(M * kvw));
    std::vector<int32_t> pos((size_t)M), set((size_t)M);
    for (int64_t m = 0; m < M; ++m) {
        int32_t id = ids[m];
        if (id < 0 || id >= D.V) return -1;
        std::memcpy(&x[(size_t)(m * D.d)], w->embed + (int64_t)id * D.d, (size_t)D.d * 2);
        pos[m] = (int32_t)(len0 + m % T);
        set[m] = (int32_t)(m / T);
    }
    int64_t layer_elems = (int64_t)B * D.hkv * cap * D.dh;
    for (int l = 0; l < D.L; ++l) {
        if (l == tap_layer && tap_in) std::memcpy(tap_in, x.data(), x.size() * 2);
        oracle_layer_qkv(c, w, l, x.data(), pos.data(), M, q.data(), k.data(), v.data());
        uint16_t* kl = kc + l * layer_elems;
        uint16_t* vl = vc + l * layer_elems;
        for (int64_t m = 0; m < M; ++m)
            for (int j = 0; j < D.hkv; ++j) {
                int64_t slot = (((int64_t)set[m] * D.hkv + j) * cap + pos[m]) * D.dh;
                std::memcpy(kl + slot, &k[(size_t)(m * kvw + (int64_t)j * D.dh)], (size_t)D.dh * 2);
                std::memcpy(vl + slot, &v[(size_t)(m * kvw + (int64_t)j * D.dh)], (size_t)D.dh * 2);
            }
        oracle_layer_out(c, w, l, x.data(), q.data(), pos.data(), M, kl, vl, set.data(), cap, y.data());
        x.swap(y);
        if (l == tap_layer && tap_out) std::memcpy(tap_out, x.data(), x.size() * 2);
    }
    if (all_rows) {
        oracle_head(c, w, x.data(), M, logits);
    } else {
        std::vector<uint16_t> last((size_t)B * D.d);
        for (int b = 0; b < B; ++b)
            std::memcpy(&last[(size_t)b * D.d], &x[(size_t)(((int64_t)b * T + T - 1) * D.d)], (size_t)D.d * 2);
        oracle_head(c, w, last.data(), B, logits);
    }
    return 0;
}

// The general form of the forward pass ("A modern architecture: Qwen3", section The whole model,
// hidden(ids, positions, mask, caches), as its batched generation section drives it): token
// r = b*T + t is rotated at position pos[r], writes its key and value into slot slot[r] of
// sequence b's cache, and then attends to the slots of sequence b that mask[r][0..cap) admits.
// Left padding, a shared prefix, a banded (sliding-window) mask and a rolling buffer are all
// choices of pos, slot and mask; this function only carries them out.
// Returns 0, -1 on a bad token id, -2 on a slot outside [0, cap), -3 on a row admitting no key.
int oracle_forward_masked(const oracle_config* c, const oracle_weights* w, uint16_t* kc, uint16_t* vc,
                          int B, int64_t cap, const int32_t* ids, int T, const int32_t* pos,
                          const int32_t* slot, const uint8_t* mask, int all_rows, float* logits,
                          int tap_layer, uint16_t* tap_in, uint16_t* tap_out) {
    Dims D(c);
    int64_t M = (int64_t)B * T;
    int64_t kvw = (int64_t)D.hkv * D.dh;
    std::vector<uint16_t> x((size_t)(M * D.d)), y((size_t)(M * D.d)), q((size_t)(M * D.hq * D.dh)),
        k((size_t)(M * kvw)), v((size_t)(M * kvw));
    std::vector<int32_t> set((size_t)M);
    for (int64_t m = 0; m < M; ++m) {
        int32_t id = ids[m];
        if (id < 0 || id >= D.V) return -1;
        if (slot[m] < 0 || slot[m] >= cap) return -2;
        std::memcpy(&x[(size_t)(m * D.d)], w->embed + (int64_t)id * D.d, (size_t)D.d * 2);
        set[m] = (int32_t)(m / T);
    }
    int64_t layer_elems = (int64_t)B * D.hkv * cap * D.dh;
    for (int l = 0; l < D.L; ++l) {
        if (l == tap_layer && tap_in) std::memcpy(tap_in, x.data(), x.size() * 2);
        oracle_layer_qkv(c, w, l, x.data(), pos, M, q.data(), k.data(), v.data());
        uint16_t* kl = kc + l * layer_elems;
        uint16_t* vl = vc + l * layer_elems;
        for (int64_t m = 0; m < M; ++m)
            for (int j = 0; j < D.hkv; ++j) {
                int64_t at = (((int64_t)set[m] * D.hkv + j) * cap + slot[m]) * D.dh;
                std::memcpy(kl + at, &k[(size_t)(m * kvw + (int64_t)j * D.dh)], (size_t)D.dh * 2);
                std::memcpy(vl + at, &v[(size_t)(m * kvw + (int64_t)j * D.dh)], (size_t)D.dh * 2);
            }
        int rc = oracle_layer_out_masked(c, w, l, x.data(), q.data(), M, kl, vl, set.data(), cap, mask, y.data());
        if (rc != 0) return rc;
        x.swap(y);
        if (l == tap_layer && tap_out) std::memcpy(tap_out, x.data(), x.size() * 2);
    }
    if (all_rows) {
        oracle_head(c, w, x.data(), M, logits);
    } else {
        std::vector<uint16_t> last((size_t)B * D.d);
        for (int b = 0; b < B; ++b)
            std::memcpy(&last[(size_t)b * D.d], &x[(size_t)(((int64_t)b * T + T - 1) * D.d)], (size_t)D.d * 2);
        oracle_head(c, w, last.data(), B, logits);
    }
    return 0;
}

}  // extern "C"
