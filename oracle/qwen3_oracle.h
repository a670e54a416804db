/*
 * Qwen3 decoder oracle: C interface.
 *
 * TEST INFRASTRUCTURE ONLY. This is a plain, slow, single-threaded CPU statement of the
 * forward pass of a Qwen3-style dense decoder, written from the pages' definitions. Only the
 * tests, the smoke check and the benchmark's CPU-baseline leg may load it. It shares no code,
 * header, table or constant with the CUDA library, and the CUDA library never calls it.
 *
 * Storage follows the model: every activation and weight is bfloat16, held here as its raw
 * 16-bit pattern (uint16_t). Each operation is evaluated exactly (fp64) and rounded once,
 * round-to-nearest-even, to the dtype the pages' PyTorch code stores it in, at exactly the
 * cast points they state:
 *   - RMSNorm: reduction and scaling in fp32, cast to bf16, THEN times gamma
 *     ("A modern architecture: Qwen3", section RMSNorm, parity detail 2;
 *      the Qwen3 checklist page, item "RMSNorm computes in float32").
 *   - RoPE: fp32 inverse frequencies and fp32 angles, cos/sin cast to bf16, the rotation
 *     x*cos + rotate_half(x)*sin evaluated op by op in bf16 ("A modern architecture: Qwen3",
 *     section Rotary position embeddings; the checklist item on the rotate-half pairing).
 *   - Linear layers, attention output, SiLU, products and residual adds: exact value, one
 *     bf16 rounding. LM-head logits stay fp32.
 *
 * Weight layout: nn.Linear [out, in] row-major; norms [n]; embedding [V, d].
 * KV cache layout: [L][B][Hkv][cap][dh], slot index = absolute position.
 *
 * Parity status of each function is stated in the source file next to it.
 */
#ifndef QWEN3_ORACLE_H
#define QWEN3_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int32_t n_layers, hidden, n_q_heads, n_kv_heads, head_dim, intermediate, vocab, tie_embeddings;
    double rope_theta, rms_eps;
} oracle_config;

/* Per-layer arrays hold n_layers host pointers each. lm_head is ignored when tie_embeddings. */
typedef struct {
    const uint16_t *embed, *lm_head, *final_norm;
    const uint16_t *const *in_norm, *const *q_proj, *const *k_proj, *const *v_proj, *const *o_proj,
                   *const *q_norm, *const *k_norm, *const *post_norm,
                   *const *gate_proj, *const *up_proj, *const *down_proj;
} oracle_weights;

/* ---- scalar conversions ---- */
uint16_t oracle_bf16_from_f32(float x);
uint16_t oracle_bf16_from_f64(double x);
float oracle_f32_from_bf16(uint16_t h);

/* ---- RMSNorm ---- */
/* fp32 core without gain or casts: y = x * rsqrt(mean(x^2) + eps). */
void oracle_rmsnorm_core_f32(const float* x, int n, double eps, float* y);
/* Qwen3 order on bf16 rows: y = bf16(gamma * bf16(core(x))). */
void oracle_rmsnorm(const uint16_t* x, const uint16_t* gamma, int64_t rows, int n, double eps, uint16_t* y);

/* ---- linear, y = a W^T ---- */
void oracle_linear(const uint16_t* a, const uint16_t* w, int64_t M, int64_t N, int64_t K, uint16_t* y);
void oracle_linear_f32out(const uint16_t* a, const uint16_t* w, int64_t M, int64_t N, int64_t K, float* y);

/* ---- residual add: out = bf16(x + y) ---- */
void oracle_residual_add(const uint16_t* x, const uint16_t* y, int64_t n, uint16_t* out);

/* ---- SwiGLU ---- */
double oracle_silu(double z);
/* a = bf16(bf16(silu(g)) * u), elementwise. */
void oracle_swiglu(const uint16_t* g, const uint16_t* u, int64_t n, uint16_t* a);

/* ---- RoPE ---- */
/* inv[i] = fp32(theta^(-2i/dim)), i < dim/2. */
void oracle_rope_inv_freq(double theta, int dim, float* inv);
/* bf16 cos/sin tables at one position: ang = fp32(pos * inv[i]). */
void oracle_rope_cos_sin(int64_t pos, const float* inv, int half, uint16_t* cos_out, uint16_t* sin_out);
/* rotate-half in bf16 arithmetic, in place on one head vector of length dim. */
void oracle_rope_apply(uint16_t* x, int dim, const uint16_t* cos_t, const uint16_t* sin_t);
/* fp64 rotate-half of one vector at position pos with explicit per-pair frequencies omega[dim/2]. */
void oracle_rope_rotate_f64(const double* x, int dim, double pos, const double* omega, double* y);

/* ---- attention ---- */
/* One query row against n keys (already selected: causal prefix or whole cache), fp64 output. */
void oracle_attention_row_f64(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t n,
                              int dim, int64_t kv_stride, double scale, double* out);
/* All query heads of one row, q [Hq][dh], against keys 0..n-1 of one cache set kc/vc
   [Hkv][cap][dh]; query head h reads kv head h / (Hq/Hkv). out [Hq][dh] in fp64. */
void oracle_attention_gqa_row_f64(const uint16_t* q, const uint16_t* kc, const uint16_t* vc, int64_t n,
                                  int hq, int hkv, int dim, int64_t cap, double* out);

/* ---- model pieces ---- */
/* Parameter count by part: [embedding, attention, qk-norm, feed-forward, other norms, lm_head]. */
void oracle_param_count(const oracle_config* c, int64_t parts[6]);

/* Steps a2-a4 for n rows of one layer: xin [n][d] is the layer input at absolute positions pos[n].
   Outputs q [n][Hq][dh] (after q_norm and RoPE), k [n][Hkv][dh] (after k_norm and RoPE),
   v [n][Hkv][dh] (raw projection). */
void oracle_layer_qkv(const oracle_config* c, const oracle_weights* w, int layer, const uint16_t* xin,
                      const int32_t* pos, int64_t n, uint16_t* q, uint16_t* k, uint16_t* v);

/* Steps a5-a9 for n rows of one layer, given the rows' queries and a KV cache view.
   Row r attends to slots 0..pos[r] of kv set kvset[r]; kc/vc are [nsets][Hkv][cap][dh].
   xout [n][d] is the layer output. */
void oracle_layer_out(const oracle_config* c, const oracle_weights* w, int layer, const uint16_t* xin,
                      const uint16_t* q, const int32_t* pos, int64_t n, const uint16_t* kc,
                      const uint16_t* vc, const int32_t* kvset, int64_t cap, uint16_t* xout);

/* Final RMSNorm and LM head for n rows: logits [n][V] fp32. */
void oracle_head(const oracle_config* c, const oracle_weights* w, const uint16_t* x, int64_t n, float* logits);

/* Whole forward pass of T new tokens for B equal-length sequences, starting at position len0,
   appending to the cache kc/vc ([L][B][Hkv][cap][dh]). ids [B*T], row-major by sequence.
   logits: [B*T][V] when all_rows, else [B][V] for each sequence's last row.
   When tap_layer >= 0, tap_in/tap_out receive that layer's input and output rows [B*T][d].
   Returns 0, or -1 on a bad token id, -2 on capacity overflow. */
int oracle_forward(const oracle_config* c, const oracle_weights* w, uint16_t* kc, uint16_t* vc,
                   int B, int64_t cap, int64_t len0, const int32_t* ids, int T, int all_rows,
                   float* logits, int tap_layer, uint16_t* tap_in, uint16_t* tap_out);

/* Masked attention of one row: q [Hq][dh] against the slots of kc/vc [Hkv][cap][dh] that
   mask[0..cap) admits (nonzero), in slot order. Returns -3 when the mask admits nothing. */
int oracle_attention_masked_gqa_row_f64(const uint16_t* q, const uint16_t* kc, const uint16_t* vc,
                                        int64_t cap, const uint8_t* mask, int hq, int hkv, int dim,
                                        double* out);

/* Steps a5-a9 with an explicit mask: row r reads the slots of kv set kvset[r] that mask[r][cap]
   admits. Returns 0 or -3 (a row admitting no key). */
int oracle_layer_out_masked(const oracle_config* c, const oracle_weights* w, int layer, const uint16_t* xin,
                            const uint16_t* q, int64_t n, const uint16_t* kc, const uint16_t* vc,
                            const int32_t* kvset, int64_t cap, const uint8_t* mask, uint16_t* xout);

/* General forward pass: token r = b*T + t is rotated at position pos[r], writes its K/V into slot
   slot[r] of sequence b's cache kc/vc ([L][B][Hkv][cap][dh]) and attends to the slots that
   mask[r][cap] admits. Left padding, a shared prefix, a sliding window and a rolling buffer are
   choices of pos, slot and mask made by the caller. Returns 0, -1 (bad token id), -2 (slot out
   of range) or -3 (a row admitting no key). */
int oracle_forward_masked(const oracle_config* c, const oracle_weights* w, uint16_t* kc, uint16_t* vc,
                          int B, int64_t cap, const int32_t* ids, int T, const int32_t* pos,
                          const int32_t* slot, const uint8_t* mask, int all_rows, float* logits,
                          int tap_layer, uint16_t* tap_in, uint16_t* tap_out);

#ifdef __cplusplus
}
#endif
#endif
