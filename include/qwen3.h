/*
 * qwen3.h - C ABI of the GB300 (sm_103a) Qwen3 decoder forward-pass library.
 *
 * The library runs the forward pass of a Qwen3-style dense decoder stack on one GPU: token
 * embedding, and per layer a pre-norm RMSNorm, Q/K/V projections (head_dim independent of
 * hidden/heads), per-head q_norm/k_norm over head_dim followed by rotate-half RoPE on Q and K,
 * causal grouped-query attention scaled by head_dim^-0.5, a residual add, RMSNorm, a SwiGLU MLP
 * and a second residual add; then a final RMSNorm and the LM head. Sources: "A modern
 * architecture: Qwen3" (sections RMSNorm, Rotary position embeddings, Attention with grouped KV
 * heads and Q/K normalization, SwiGLU, The whole model) and the Qwen3 block checklist page.
 *
 * Conventions for every call:
 *  - Pointers named d_* are device pointers; h_* are host pointers. Tensors are dense row-major.
 *  - bf16 tensors hold IEEE bfloat16; logits are fp32.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream). Calls enqueue
 *    asynchronously on it and never synchronise, except where a call says it does.
 *  - Every call returns QWEN3_OK (0) or one of the QWEN3_E_* codes below; on an error nothing has
 *    been enqueued unless stated. qwen3_strerror() names a code.
 *  - The library never falls back to the CPU: every step of the forward pass runs in its kernels.
 */
#ifndef QWEN3_H
#define QWEN3_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define QWEN3_API __attribute__((visibility("default")))
#else
#define QWEN3_API
#endif

#define QWEN3_OK 0
#define QWEN3_E_CONFIG 1     /* invalid or unsupported model shape */
#define QWEN3_E_CAPACITY 2   /* cache capacity above max_positions ("new_cache" check) */
#define QWEN3_E_OVERFLOW 3   /* length + new tokens above the cache capacity */
#define QWEN3_E_BATCH 4      /* batch or token count above what the context was sized for */
#define QWEN3_E_ARG 5        /* null pointer or out-of-range argument */
#define QWEN3_E_CUDA 6       /* CUDA launch, allocation or driver failure */
#define QWEN3_E_TOKEN 7      /* device flag: a token id was outside [0, vocab); its row was zeroed */
#define QWEN3_E_TIMEOUT 8    /* device flag: a kernel's bounded wait gave up; its output is invalid */
#define QWEN3_E_DEVICE 9     /* the current device is not an sm_103 GPU */

/* Prefill flag: return logits for every row instead of each sequence's last row. */
#define QWEN3_ALL_ROWS 1

/* Model shape. Field meanings follow the Qwen3 config (hidden_size, num_hidden_layers, ...). */
typedef struct qwen3_config {
    int32_t n_layers;       /* num_hidden_layers */
    int32_t hidden;         /* hidden_size d; multiple of 64 */
    int32_t n_q_heads;      /* num_attention_heads Hq; multiple of n_kv_heads */
    int32_t n_kv_heads;     /* num_key_value_heads Hkv */
    int32_t head_dim;       /* dh: 64 or 128 (not hidden / heads in general) */
    int32_t intermediate;   /* intermediate_size F; multiple of 128 */
    int32_t vocab;          /* vocab_size V; multiple of 8 */
    int32_t tie_embeddings; /* nonzero: LM head reuses the embedding matrix */
    int32_t max_positions;  /* max_position_embeddings: upper bound for the cache capacity */
    float rope_theta;       /* RoPE base theta (1e6 for Qwen3) */
    float rms_eps;          /* RMSNorm epsilon (1e-6 for Qwen3) */
    /* Sliding-window attention ("A modern architecture: Qwen3", section 7): 0 = full causal
     * attention (Qwen3); W > 0 = in every layer the token in slot i sees slots j with i - W < j <= i. */
    int32_t sliding_window;
    /* With a window: 0 = the cache keeps every slot (the banded mask over a full cache); 1 = a
     * rolling buffer that stores slot s at s mod R, R = W + min(ceil(max_tokens / max_batch),
     * capacity) - 1 rounded up to 256, so the cache holds R slots per sequence and head however long
     * the sequence grows.
     * Prefill calls then take at most R - W + 1 tokens per sequence (E_BATCH beyond). */
    int32_t rolling_cache;
} qwen3_config;

/* Device pointers to bf16 weights, BORROWED: they must stay valid until qwen3_free(). Linear
 * weights use the nn.Linear layout [out, in]. Per-layer fields point to arrays of n_layers device
 * pointers held in HOST memory (the arrays are read during qwen3_init only). */
typedef struct qwen3_weights {
    const void* embed;       /* [V, d] */
    const void* lm_head;     /* [V, d]; ignored (may be NULL) when tie_embeddings */
    const void* final_norm;  /* [d] */
    const void* const* in_norm;    /* [d]          input_layernorm */
    const void* const* q_proj;     /* [Hq*dh, d] */
    const void* const* k_proj;     /* [Hkv*dh, d] */
    const void* const* v_proj;     /* [Hkv*dh, d] */
    const void* const* o_proj;     /* [d, Hq*dh] */
    const void* const* q_norm;     /* [dh]         shared by all query heads */
    const void* const* k_norm;     /* [dh]         shared by all kv heads */
    const void* const* post_norm;  /* [d]          post_attention_layernorm */
    const void* const* gate_proj;  /* [F, d] */
    const void* const* up_proj;    /* [F, d] */
    const void* const* down_proj;  /* [d, F] */
} qwen3_weights;

typedef struct qwen3_ctx qwen3_ctx;

/* Host-only check of a shape (no GPU needed). Rejects Hq % Hkv != 0 ("Query heads must be a
 * multiple of KV heads", Attention section), head_dim outside {64, 128}, and sizes that break the
 * kernels' tiling (hidden % 64, intermediate % 128, vocab % 8, head counts < 1). */
QWEN3_API int qwen3_validate_config(const qwen3_config* cfg);

/* Create a context on the current device: validates the shape, checks capacity <= max_positions
 * (the "new_cache" rule), allocates and zeroes the KV cache [L][max_batch][Hkv][capacity][dh] (bf16,
 * keys stored after q/k-norm and RoPE, slot = absolute position), activation scratch for up to
 * max_tokens rows per prefill call (0 means max_batch * capacity), packed copies of the fused
 * QKV and gate/up weights, and the bf16 RoPE table [capacity][dh/2] of cos and sin.
 * The context owns everything it allocates; qwen3_free() releases it. Synchronises `stream`.
 * Errors: E_ARG, E_CONFIG, E_CAPACITY, E_CUDA (e.g. out of memory), E_DEVICE. */
QWEN3_API int qwen3_init(const qwen3_config* cfg, const qwen3_weights* w, int max_batch, int capacity,
               int max_tokens, void* stream, qwen3_ctx** out);

/* Causal prefill of T new tokens for B equal-length sequences ("forward(ids, cache, ...)", The
 * whole model section): positions are length .. length+T-1, K/V are appended to the cache at those
 * slots, and length += T. d_ids: [B*T] int32, sequence-major. d_logits: fp32 [B, V] (each
 * sequence's last row) or [B*T, V] with QWEN3_ALL_ROWS. A prefill after a previous call continues
 * every sequence from the current length. Errors: E_ARG, E_BATCH (B > max_batch, B*T > max_tokens,
 * or B differs from the batch already in the cache), E_OVERFLOW (length + T > capacity), E_CUDA. */
QWEN3_API int qwen3_prefill(qwen3_ctx* ctx, const int32_t* d_ids, int B, int T, float* d_logits, int flags,
                  void* stream);

/* One greedy-decode forward step ("A modern architecture: Qwen3", The whole model: the generation loop
 * feeds the argmax token back with positions = cache.length; "Transformer architectures: modern",
 * generation): one token per sequence at position = length, appended to the cache; length += 1.
 * d_ids: [B] int32 (B must equal the batch already in the cache); d_logits: fp32 [B, V]. The step is
 * replayed from a CUDA graph that the context captures on first use for each (B, d_ids, d_logits,
 * number of 512- or 1024-slot context chunks holding keys); kernels read the length from device memory,
 * so replays advance correctly. Errors as qwen3_prefill. */
QWEN3_API int qwen3_decode_step(qwen3_ctx* ctx, const int32_t* d_ids, int B, float* d_logits, void* stream);

/* End-to-end variant of qwen3_prefill on HOST buffers: copies h_ids to the device, runs the
 * prefill, copies the logits back to h_logits and synchronises `stream`. Host buffers should be
 * pinned for full copy bandwidth. Same errors as qwen3_prefill, plus device flags (E_TOKEN,
 * E_TIMEOUT) read after the synchronisation. */
QWEN3_API int qwen3_prefill_host(qwen3_ctx* ctx, const int32_t* h_ids, int B, int T, float* h_logits,
                       int flags, void* stream);

/* Left-padded batch prefill ("A modern architecture: Qwen3", generation with a batch of prompts):
 * row b of d_ids [B*T] holds h_real[b] real tokens (1..T, HOST array) at its end, after T - h_real[b]
 * padding tokens. Padding gets no attention from any other token, each padding token attends to
 * itself (and to every earlier real slot), and positions count real tokens: the k-th real token of
 * a row is at position length + k, padding at max(length - 1, 0). Later prefill and decode calls keep
 * the layout (each row's next position is its own count of real tokens). Allowed once per fill of
 * the cache (qwen3_set_length clears the layout); rows without padding are ordinary prefill.
 * Errors as qwen3_prefill, plus E_ARG (h_real out of range, a second padded block, or a context with
 * a sliding window). */
QWEN3_API int qwen3_prefill_padded(qwen3_ctx* ctx, const int32_t* d_ids, const int32_t* h_real, int B, int T,
                                   float* d_logits, int flags, void* stream);

/* Prefix caching ("A modern architecture: Qwen3", section 8): after a one-sequence prefill of a shared
 * start of P tokens, make it the start of B sequences without recomputing it. Whole 128-slot tiles
 * of the start are read in place from sequence 0's cache by every sequence; the remaining P mod 128
 * slots are copied into sequences 1..B-1. The batch becomes B at length P; the next call continues all
 * B sequences (qwen3_prefill_padded for prompts of different lengths). Errors: E_BATCH (B out of
 * range), E_ARG (the cache does not hold exactly one unpadded sequence, a prefix is already shared,
 * or the context has a sliding window), E_CUDA. */
QWEN3_API int qwen3_share_prefix(qwen3_ctx* ctx, int B, void* stream);

/* Greedy generation, the pages' generate loop: prefill of d_ids (left-padded by h_real when h_real
 * is not NULL, else equal-length), then up to max_new tokens per row chosen by argmax of each step's
 * logits (lowest index on ties), each fed back through qwen3_decode_step. With stop_id >= 0 a row that
 * emits stop_id is finished and emits stop_id from then on, and the loop ends when every row has
 * finished (the host reads a device counter after each step; this synchronises `stream`). Token k of
 * row b goes to d_out[b * max_new + k]; *h_steps receives the number of columns written, later columns
 * are left untouched. Errors as qwen3_prefill_padded / qwen3_decode_step, and E_OVERFLOW when the
 * cache cannot hold T + max_new - 1 more tokens. */
QWEN3_API int qwen3_generate(qwen3_ctx* ctx, const int32_t* d_ids, const int32_t* h_real, int B, int T, int max_new,
                             int stop_id, int32_t* d_out, int* h_steps, void* stream);

/* Current cache length (tokens per sequence) and batch held in the cache. */
QWEN3_API int qwen3_length(const qwen3_ctx* ctx, int* length, int* batch);

/* Set the cache length and batch ("A modern architecture: Qwen3", The whole model: the preallocated
 * KVCache and its `length`, which positions continue from), e.g. after filling the cache through
 * qwen3_kv_view. Enqueues a device update on `stream`. The cache then holds plain equal-length
 * sequences: any padding layout or shared prefix is cleared. Errors: E_ARG, E_OVERFLOW (length >
 * capacity), E_BATCH. */
QWEN3_API int qwen3_set_length(qwen3_ctx* ctx, int length, int batch, void* stream);

/* The preallocated KV cache ("A modern architecture: Qwen3", The whole model: new_cache allocates
 * K and V per layer as [batch, kv heads, capacity, head_dim]; keys are cached already rotated, Attention
 * with grouped KV heads). Device pointers to layer `layer`'s K and V cache, each [max_batch][Hkv][slots][dh] bf16,
 * dims[0..3] = {max_batch, Hkv, slots, dh}; slots = capacity, or the ring size of a rolling buffer.
 * The memory stays owned by the context. */
QWEN3_API int qwen3_kv_view(qwen3_ctx* ctx, int layer, void** d_k, void** d_v, int64_t dims[4]);

/* Debug tap: on later prefill/decode calls, copy layer `layer`'s input and output hidden states
 * ([rows, d] bf16, rows = B*T) into caller buffers sized for the largest call. layer < 0 turns
 * the tap off. Taps are copies enqueued on the call's stream; they change no result. */
QWEN3_API int qwen3_set_tap(qwen3_ctx* ctx, int layer, void* d_layer_in, void* d_layer_out);

/* Synchronise `stream`, then read and clear the device error flags: returns QWEN3_OK,
 * QWEN3_E_TOKEN or QWEN3_E_TIMEOUT (or E_CUDA if the synchronisation failed). The pages' forward pass
 * raises on invalid input ("A modern architecture: Qwen3", The whole model: the context-limit check);
 * a kernel cannot raise, so a token id outside [0, vocab) zeroes its embedding row and sets a flag that
 * this call reports. */
QWEN3_API int qwen3_get_error(qwen3_ctx* ctx, void* stream);

/* Per-kernel timing: while enabled, every kernel launch of a call is bracketed by CUDA events on
 * the call's stream. qwen3_kernel_times() synchronises the last timed stream and writes, for each
 * kernel class i < *n (classes named by qwen3_kernel_class_name), the total milliseconds and
 * launch count since timing was enabled; it then resets the totals. *n is in: capacity of the
 * arrays, out: number of classes. */
QWEN3_API int qwen3_set_timing(qwen3_ctx* ctx, int enable);
QWEN3_API int qwen3_kernel_times(qwen3_ctx* ctx, double* total_ms, int64_t* launches, int* n);
QWEN3_API const char* qwen3_kernel_class_name(int i);

/* Number of kernel launches a prefill of B x T or a decode step of B makes (for launch accounting). */
QWEN3_API int qwen3_launch_count(const qwen3_ctx* ctx, int B, int T, int flags, int decode);

/* Name of an error code (the pages' errors: head divisibility and odd rotary dimension, Attention with
 * grouped KV heads and Rotary position embeddings sections; capacity and context overflow, The whole
 * model). Returns a static string; never NULL. */
QWEN3_API const char* qwen3_strerror(int code);
/* Release a context and everything it owns (the cache the pages' new_cache allocates, scratch, packed
 * weights, captured graphs). Synchronises the device first. The borrowed weights are not touched.
 * NULL is ignored. */
QWEN3_API void qwen3_free(qwen3_ctx* ctx);

/* ------------------------------------------------------------------------------------------------
 * Single-operation entry points. Each enqueues the same kernels the forward pass uses, on caller
 * buffers, so each step can be checked on its own. All pointers are device pointers.
 * ----------------------------------------------------------------------------------------------*/

/* Embedding gather: out[m, :] = embed[ids[m], :] for m < M (embed [V, d] bf16, d % 8 == 0).
 * An id outside [0, V) zeroes its row and sets bit 1 in *d_err (device int). */
QWEN3_API int qwen3_op_embed(const void* d_embed, int V, int d, const int32_t* d_ids, int M, void* d_out,
                   int* d_err, void* stream);

/* RMSNorm, Qwen3 order (RMSNorm section, parity detail 2): y = bf16(gamma * bf16(x * rsqrt(
 * mean(x^2) + eps))), the mean and scaling in fp32. x rows are read at row index
 * r * in_stride + in_offset (r < rows), so the last row of each sequence can be normalised alone;
 * y is [rows, n]. n % 8 == 0, n <= 8192. */
QWEN3_API int qwen3_op_rmsnorm(const void* d_x, const void* d_gamma, int rows, int n, int in_stride,
                     int in_offset, float eps, void* d_y, void* stream);

/* GEMM on the tensor cores: acc = A B^T with A [M, K] and B [N, K] bf16 (nn.Linear layout),
 * fp32 accumulation; K % 8 == 0. Epilogues:
 *   QWEN3_EPI_BF16     C [M, N] bf16 = bf16(acc)
 *   QWEN3_EPI_SWIGLU   B packed by qwen3_op_pack_gate_up (N = 2F); C [M, F] bf16 =
 *                      bf16(bf16(silu(bf16(gate))) * bf16(up))        (SwiGLU section)
 *   QWEN3_EPI_RESIDUAL C [M, N] bf16 = bf16(R + bf16(acc)); R may alias C (residual add)
 *   QWEN3_EPI_F32      C [M, N] fp32 = acc                            (LM-head logits)
 * ldc / ldr are row strides in elements. d_err receives bit 2 if a bounded wait gave up. */
#define QWEN3_EPI_BF16 0
#define QWEN3_EPI_SWIGLU 1
#define QWEN3_EPI_RESIDUAL 2
#define QWEN3_EPI_F32 3
QWEN3_API int qwen3_op_gemm(const void* d_A, const void* d_B, int M, int N, int K, int epilogue, void* d_C,
                  int ldc, const void* d_R, int ldr, int* d_err, void* stream);

/* Residual GEMM fused with the next RMSNorm (the pre-norm block: each residual add is followed by
 * the next sub-layer's RMSNorm): X [M, N] bf16 (row stride N) is updated in place to
 * bf16(X + bf16(A B^T)), then Y [M, N] bf16 = bf16(gamma * bf16(X * rsqrt(mean(X^2) + eps))) over
 * each full updated row, the mean in fp32. The N / BN column tiles of a row block (BN = 128 or 256,
 * the tile width the library picks for [M, N]) run concurrently in one cooperative launch and
 * exchange per-row partial sums; qwen3_gemm_norm_supported says whether a shape qualifies (N a
 * multiple of the tile width, at most 8 tiles). d_part is scratch of qwen3_gemm_norm_part_floats(M)
 * 4-byte words, zeroed before the first call and otherwise left to the library (each call leaves its
 * counters zero; after a call that set d_err, zero it again). Returns QWEN3_E_ARG for an unsupported
 * shape; d_err receives bit 2 if a bounded wait gave up. */
QWEN3_API int qwen3_gemm_norm_supported(int M, int N);
QWEN3_API size_t qwen3_gemm_norm_part_floats(int M);
QWEN3_API int qwen3_op_gemm_residual_norm(const void* d_A, const void* d_B, int M, int N, int K, void* d_X,
                                          const void* d_gamma, float eps, void* d_Y, float* d_part, int* d_err,
                                          void* stream);

/* Weight-streaming GEMM for a few rows (decode batches, 1 <= M <= 64): acc[b][n] = sum_k A[b][k] B[n][k]
 * in fp32 on the tensor cores, with the weights B [N, K] as the 128-row MMA operand and the K range
 * split over `splits` CTAs per 128 weight rows (qwen3_gemm_skinny_splits gives the runtime's choice).
 * splits == 1: d_out [M, N] fp32 receives acc. splits > 1: d_slices receives split s's partial sums
 * at [s][M][N] fp32 (splits * M * N floats); their sum is acc. K % 8 == 0. */
QWEN3_API int qwen3_gemm_skinny_splits(int N, int K);
QWEN3_API int qwen3_op_gemm_skinny(const void* d_A, const void* d_B, int M, int N, int K, int splits, float* d_slices,
                                   float* d_out, int* d_err, void* stream);

/* Pack gate [F, d] and up [F, d] into the [2F, d] layout QWEN3_EPI_SWIGLU expects: blocks of 128
 * gate rows followed by the matching 128 up rows. F % 128 == 0. */
QWEN3_API int qwen3_op_pack_gate_up(const void* d_gate, const void* d_up, int F, int d, void* d_out, void* stream);

/* RoPE table: cos_sin [n_pos][dh] bf16, row p = (cos(p w_0..), sin(p w_0..)) for the dh/2 pair
 * frequencies w_i = fp32(theta^(-2i/dh)), angle = fp32(p * w_i), each cos/sin rounded from fp32 to
 * bf16 (Rotary position embeddings section: rope_cos_sin). */
QWEN3_API int qwen3_op_rope_table(float theta, int dh, int n_pos, void* d_cos_sin, void* stream);

/* Fused q_norm / k_norm + RoPE + KV-cache append (Attention section: q and k are normalised per
 * head over head_dim, then rotated; V passes untouched; keys are cached already rotated).
 * qkv: [B*T, (Hq + 2 Hkv) dh] bf16 rows (q heads, then k heads, then v heads), positions
 * len0 + t. Writes Q to q_out [B, Hq, T, dh] and K/V to k_cache/v_cache [B, Hkv, cap, dh] at slot
 * len0 + t. len0 is read from *d_len0 (device int) so graph replays see the current length. */
QWEN3_API int qwen3_op_qknorm_rope_append(const void* d_qkv, int B, int T, int Hq, int Hkv, int dh,
                                const void* d_q_gamma, const void* d_k_gamma, const void* d_cos_sin,
                                const int* d_len0, float eps, void* d_q_out, void* d_k_cache,
                                void* d_v_cache, int cap, void* stream);

/* Causal GQA attention for prefill: for query row t of sequence b (cache slot len0 + t) and query
 * head h, out = softmax(q k^T * dh^-0.5 over cache slots 0..len0+t of kv head h / (Hq/Hkv)) V.
 * d_seq_meta (may be NULL) gives a padding layout and shared prefix as qwen3_prefill_padded and
 * qwen3_share_prefix build it: ints [ps, psh, pad_0 .. pad_{B-1}]; slots [ps, ps + pad_b) of sequence b
 * are seen only by themselves, slots below psh (a multiple of 128) are read from sequence 0.
 * window > 0 restricts slot i to keys j > i - window; ring > 0 (= cap, a multiple of 256, with a
 * window) reads slot s from cache row s mod ring. heads_per_cta: query heads of one kv group per CTA (1 or 2,
 * 2 needs an even group size; 0 = the forward pass's choice).
 * q [B, Hq, T, dh]; caches [B, Hkv, cap, dh] with len0 + T <= cap; out [B*T, Hq*dh] bf16
 * (token-major, the o_proj input). kv_split > 0 cuts each 128-row query tile's key range into at most
 * kv_chunks chunks of at least kv_split 128-key tiles, computed by separate CTAs and merged by
 * log-sum-exp in the last one to finish; d_work then holds qwen3_attention_prefill_workspace() bytes
 * whose first 256 bytes are zero on the first call (each call leaves them zero). kv_split = 0: one CTA
 * per query tile, d_work unused. d_err (may be NULL) receives bit 2 if a bounded wait gave up. */
QWEN3_API size_t qwen3_attention_prefill_workspace(int B, int T, int Hq, int Hkv, int dh, int kv_chunks);
QWEN3_API int qwen3_op_attention_prefill(const void* d_q, const void* d_k_cache, const void* d_v_cache, int B,
                               int T, int Hq, int Hkv, int dh, int cap, const int* d_len0, const int* d_seq_meta,
                               int window, int ring, int heads_per_cta, int kv_split, int kv_chunks, void* d_work,
                               void* d_out, int* d_err, void* stream);

/* Decode attention ("A modern architecture: Qwen3", Attention with grouped KV heads; the decode loop of
 * The whole model): one query per (b, h) against cache slots 0..n-1, n = *d_len0 + 1, kv head
 * h / (Hq/Hkv), split over the context in chunks and merged by log-sum-exp. q [B, Hq, dh]; out
 * [B, Hq*dh] bf16. d_seq_meta, window and ring as for qwen3_op_attention_prefill (padding slots are
 * skipped, a window keeps the last `window` slots, a ring wraps; ring > 0 must be a multiple of 256).
 * d_work is caller scratch of qwen3_attention_decode_workspace(B, Hq, dh, cap, window, ring) bytes; its
 * contents on entry do not matter (a call writes every record it reads back and reads only those).
 * Caches [B, Hkv, cap, dh] bf16 with 16-byte aligned bases (they are read through TMA tensor maps; a
 * base the map rejects returns QWEN3_E_CUDA). Scores and the weighted sum run on the tensor cores with
 * fp32 accumulation; the probabilities are rounded to bf16 for the weighted sum, as in the prefill.
 * d_err (device int, may be NULL) receives bit 2 if a bounded wait gave up; the output is then invalid. */
QWEN3_API size_t qwen3_attention_decode_workspace(int B, int Hq, int dh, int cap, int window, int ring);
QWEN3_API int qwen3_op_attention_decode(const void* d_q, const void* d_k_cache, const void* d_v_cache, int B,
                              int Hq, int Hkv, int dh, int cap, const int* d_len0, const int* d_seq_meta,
                              int window, int ring, void* d_work, void* d_out, int* d_err, void* stream);

/* Greedy next token ("A modern architecture: Qwen3", generation): next[b] = the index of the largest
 * of the V fp32 logits in row b (row stride ld floats; the lowest index on ties, a NaN counting as the
 * largest, as torch.argmax). With stop_id >= 0 and d_done (int [B], device): a row with done[b] != 0
 * emits stop_id, and done[b] becomes 1 once the row emits stop_id. V % 4 == 0, ld % 4 == 0, logits
 * 16-byte aligned. d_work (may be NULL) is scratch of qwen3_greedy_workspace(B) bytes, 16-byte aligned,
 * zero before its first use (each call leaves it as the next call needs it); with it each row is split
 * over several CTAs and merged by the last one to finish, without it one CTA reads each row. Calls that
 * share a d_work must not overlap on the GPU. */
QWEN3_API size_t qwen3_greedy_workspace(int B);
QWEN3_API int qwen3_op_greedy(const float* d_logits, int64_t ld, int B, int V, int stop_id, int32_t* d_done,
                              int32_t* d_next, int32_t* d_work, void* stream);

/* Allocation-free variant of qwen3_op_attention_decode, for callers that cannot call cudaMalloc:
 * code whose device memory belongs to another allocator (for example a framework's caching pool),
 * code that must not trigger the device-wide synchronisation an allocation can cause, and code that
 * may not allocate once it has started. Same arguments and result as qwen3_op_attention_decode,
 * minus the workspace and the sequence layout (plain causal sequences only): the split partials go to a
 * fixed array compiled into this library, QWEN3_DECODE_NOALLOC_MAX_BYTES (16 MiB) large, which every GPU
 * that loads the library holds until the process exits. A call whose workspace
 * (qwen3_attention_decode_workspace(B, Hq, dh, cap, 0, 0)) is larger returns QWEN3_E_ARG and launches
 * nothing. The call allocates nothing itself. Its first call on each device looks up the array's device
 * address with that device current and keeps it for the life of the process; make that first call
 * before any stream capture, and do not call it again on a device after that device was reset
 * (cudaDeviceReset), since the kept address then no longer names the array. All calls on a device share
 * the one array and it keeps the last call's contents: calls that overlap on the GPU (other streams,
 * concurrent graph launches) race and corrupt each other's results, so serialise them. The array needs
 * no clearing: a call reads back only the partials it wrote itself (the merge skips the records of
 * chunks past the current length and the output floats of records with no visible key), so what a
 * previous call left there, even NaN or infinity, cannot reach the output.
 * d_err as for qwen3_op_attention_decode. The pages have no counterpart to this entry point. */
#define QWEN3_DECODE_NOALLOC_MAX_BYTES (16u << 20)
QWEN3_API int qwen3_op_attention_decode_noalloc(const void* d_q, const void* d_k_cache, const void* d_v_cache, int B,
                                                int Hq, int Hkv, int dh, int cap, const int* d_len0, void* d_out,
                                                int* d_err, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* QWEN3_H */
