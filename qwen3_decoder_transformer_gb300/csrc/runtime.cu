// Runtime behind the C ABI (include/qwen3.h): context ownership, shape validation, the per-layer
// launch sequence of the forward pass ("A modern architecture: Qwen3", The whole model: embed,
// L pre-norm blocks, final norm, LM head; positions continue from the cache length), CUDA-graph
// replay of decode steps, per-kernel event timing, and the single-operation entry points.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/qwen3.h"
#include "internal.h"

using bf16 = __nv_bfloat16;
using namespace q3;

namespace {

enum KernelClass : int {
    K_EMBED = 0,
    K_RMSNORM,
    K_GEMM_QKV,
    K_ATTN_PREFILL,
    K_GEMM_O,
    K_GEMM_GATEUP,
    K_GEMM_DOWN,
    K_GEMM_LMHEAD,
    K_ATTN_DECODE,
    K_LENGTH,
    K_FINALIZE,
    K_NUM_CLASSES
};
const char* kClassNames[K_NUM_CLASSES] = {"embed",
                                          "rmsnorm",
                                          "gemm_qkv_norm_rope_append",
                                          "attn_prefill",
                                          "gemm_o_residual",
                                          "gemm_gateup_swiglu",
                                          "gemm_down_residual",
                                          "gemm_lmhead",
                                          "attn_decode",
                                          "length_update",
                                          "decode_finalize"};

struct TimedLaunch {
    int cls;
    int launches;
    cudaEvent_t start, stop;
};

// A captured forward pass. Everything the host decides for a call is in the key: the shape, the
// flags, the device buffers baked into the launches, and the cache length's effect on the grids (prefill:
// the length, which picks the attention split; decode: the number of context chunks holding keys, which
// sizes the decode-attention grid, so a decode graph is reused until the length crosses a chunk boundary);
// the cache length itself, the sequence layout and the weights are read on the device.
struct ForwardGraph {
    int B, T, flags, decode, len;
    const int32_t* ids;
    float* logits;
    cudaGraphExec_t exec;
};
constexpr size_t kMaxGraphs = 16;  // oldest captured pass is dropped beyond this

bool is_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

namespace q3 {
cudaError_t prepare_kernels() {
    static std::mutex mu;
    static bool done[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev]) return cudaSuccess;
    cudaError_t e = gemm_prepare();
    if (e == cudaSuccess) e = attention_prepare();
    if (e == cudaSuccess) done[dev] = true;
    return e;
}
}  // namespace q3

struct qwen3_ctx {
    qwen3_config cfg;
    int max_batch = 0, capacity = 0, max_tokens = 0;
    // physical cache slots per (sequence, kv head): capacity, or the rolling buffer's ring
    int slots = 0, window = 0, ring = 0;
    int qkv_n = 0, q_width = 0;
    // borrowed weights
    const bf16 *embed = nullptr, *head = nullptr, *final_norm = nullptr;
    std::vector<const bf16*> in_norm, q_norm, k_norm, post_norm, o_proj, down_proj;
    // owned device memory
    bf16 *wqkv = nullptr, *wgu = nullptr, *kcache = nullptr, *vcache = nullptr, *rope = nullptr;
    bf16 *x = nullptr, *xn = nullptr, *q = nullptr, *attn = nullptr, *h = nullptr, *hn = nullptr;
    float* dec_work = nullptr;
    float* skinny_ws = nullptr;  // decode split-K GEMM accumulator [64][max N] fp32, kept zero between uses
    float* fin_part = nullptr;   // decode residual + RMSNorm: per-(row, chunk) partial sums of squares
    int* fin_tick = nullptr;     // and per-row tickets (zero between launches)
    long long skinny_ld = 0;
    CUtensorMap tX_xn, tX_attn, tX_h, tX_hn;  // decode activation maps (64-row boxes)
    float* attn_ws = nullptr;  // split prefill attention: tickets + partials (zeroed at init)
    size_t attn_ws_bytes = 0;
    int* d_len = nullptr;
    int* d_err = nullptr;
    // sequence layout (SeqMap::meta): [ps, psh, pad[0..max_batch)], with its host mirror
    int* d_seq = nullptr;
    std::vector<int> h_seq;
    bool padded = false;
    // greedy generation state: logits of the last rows, finished flags, next ids, running count
    float* gen_logits = nullptr;
    int *gen_done = nullptr, *gen_next = nullptr, *gen_alive = nullptr;
    int* gen_work = nullptr;  // greedy kernel: per-row tickets (zero between launches) and candidates
    int* h_alive = nullptr;  // pinned
    int32_t* d_ids_buf = nullptr;
    float* d_logits_buf = nullptr;
    size_t logits_buf_elems = 0;
    size_t layer_elems = 0;
    // host mirror of the cache state
    int len = 0, batch = 0;
    // tensor maps: A operands (activation buffers) and B operands (weights) per layer
    CUtensorMap tA_xn, tA_attn, tA_h, tA_hn;
    CUtensorMap tC_x, tC_h;  // staged-epilogue outputs: residual stream (also the residual input), SwiGLU output
    CUtensorMap tC_xn;       // normalised rows written by the fused residual + RMSNorm epilogue
    float* norm_part = nullptr;     // its per-row partial sums of squares
    unsigned* norm_count = nullptr;  // and the row blocks' meeting counters (zero between launches)
    std::vector<CUtensorMap> tB_qkv, tB_o, tB_gu, tB_down;
    std::vector<CUtensorMap> tK3, tV3;  // per-layer cache maps [max_batch*Hkv][cap][dh] for the fused QKV stores
    CUtensorMap tB_head;
    // captured forward passes (replayed when a call repeats)
    std::vector<ForwardGraph> graphs;
    cudaStream_t cap_stream = nullptr;
    // timing
    bool timing = false;
    std::vector<TimedLaunch> timed;
    std::vector<cudaEvent_t> free_events;
    cudaStream_t last_timed = nullptr;  // may be the legacy default stream (null handle)
    bool have_timed = false;
    // debug tap
    int tap_layer = -1;
    void *tap_in = nullptr, *tap_out = nullptr;
};

namespace {

cudaEvent_t take_event(qwen3_ctx* c) {
    if (!c->free_events.empty()) {
        cudaEvent_t e = c->free_events.back();
        c->free_events.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

// Launch `fn` (returning cudaError_t) on st; with timing on, bracket it with events.
template <typename F>
int timed(qwen3_ctx* c, int cls, int launches, cudaStream_t st, F&& fn) {
    cudaEvent_t a = nullptr, b = nullptr;
    if (c->timing) {
        a = take_event(c);
        b = take_event(c);
        cudaEventRecord(a, st);
    }
    cudaError_t e = fn();
    if (c->timing) {
        cudaEventRecord(b, st);
        c->timed.push_back({cls, launches, a, b});
        c->last_timed = st;
        c->have_timed = true;
    }
    return e == cudaSuccess ? QWEN3_OK : QWEN3_E_CUDA;
}

#define TRY(x)                              \
    do {                                    \
        int _rc = (x);                      \
        if (_rc != QWEN3_OK) return _rc;    \
    } while (0)

int gemm(qwen3_ctx* c, int cls, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap* tc,
         const CUtensorMap* tr, int M, int N, int K, int epi, void* C, long long ldc, const bf16* R, long long ldr,
         cudaStream_t st) {
    GemmArgs a{M, N, K, epi, 1, C, ldc, R, ldr, c->d_err, {}};
    GemmMaps m;
    std::memset(&m, 0, sizeof(m));
    m.a = ta;
    m.b = tb;
    if (tc) m.c = *tc;
    if (tr) m.r = *tr;
    return timed(c, cls, 1, st, [&] { return gemm_launch(m, a, st); });
}

// Residual GEMM (x += A B^T) whose epilogue also writes xn = RMSNorm(x; gamma), see EPI_RESIDUAL_NORM.
int gemm_norm(qwen3_ctx* c, int cls, const CUtensorMap& ta, const CUtensorMap& tb, int M, int N, int K,
              const bf16* gamma, cudaStream_t st) {
    GemmArgs a{M, N, K, EPI_RESIDUAL_NORM, 1, c->x, N, c->x, N, c->d_err, {},
               NormArgs{gamma, c->cfg.rms_eps, c->norm_part, c->norm_count}};
    GemmMaps m;
    std::memset(&m, 0, sizeof(m));
    m.a = ta;
    m.b = tb;
    m.c = c->tC_x;
    m.r = c->tC_x;
    m.v = c->tC_xn;
    return timed(c, cls, 1, st, [&] { return gemm_launch(m, a, st); });
}

bf16* layer_k(qwen3_ctx* c, int l) { return c->kcache + (size_t)l * c->layer_elems; }
SeqMap seq_map(const qwen3_ctx* c) { return SeqMap{c->d_seq, c->window, c->ring}; }
bf16* layer_v(qwen3_ctx* c, int l) { return c->vcache + (size_t)l * c->layer_elems; }

int skinny(qwen3_ctx* c, int cls, const CUtensorMap& tw, const CUtensorMap& tx, int M, int N, int K, float* out,
           int splits, cudaStream_t st) {
    SkinnyArgs a{M, N, K, splits, c->skinny_ws, N, out, N, c->d_err, 1};
    return timed(c, cls, 1, st, [&] { return gemm_skinny_launch(tw, tx, a, st); });
}

// Decode step for B <= 64 sequences: weight-streaming split-K GEMMs into per-split fp32 slices, each
// followed by a finalize kernel that adds the slices in order and applies the epilogue (q/k-norm +
// RoPE + cache append, residual add fused with the next RMSNorm, SwiGLU).
int enqueue_decode_skinny(qwen3_ctx* c, const int32_t* ids, int B, float* logits, cudaStream_t st) {
    const qwen3_config& g = c->cfg;
    const int d = g.hidden, dh = g.head_dim, F = g.intermediate, L = g.n_layers;
    const int s_qkv = skinny_splits(c->qkv_n, d), s_o = skinny_splits(d, c->q_width);
    const int s_gu = skinny_splits(2 * F, d), s_dn = skinny_splits(d, F);
    TRY(timed(c, K_EMBED, 1, st, [&] { return embed_launch(c->embed, g.vocab, d, ids, B, c->x, c->d_err, st); }));
    TRY(timed(c, K_RMSNORM, 1, st, [&] { return rmsnorm_launch(c->x, c->in_norm[0], B, d, 1, 0, g.rms_eps, c->xn, st); }));
    for (int l = 0; l < L; ++l) {
        if (l == c->tap_layer && c->tap_in)
            if (cudaMemcpyAsync(c->tap_in, c->x, (size_t)B * d * 2, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
                return QWEN3_E_CUDA;
        TRY(skinny(c, K_GEMM_QKV, c->tB_qkv[l], c->tX_xn, B, c->qkv_n, d, nullptr, s_qkv, st));
        TRY(timed(c, K_FINALIZE, 1, st, [&] {
            return qknorm_rope_append_f32_launch(c->skinny_ws, s_qkv, B, g.n_q_heads, g.n_kv_heads, dh, c->q_norm[l],
                                                 c->k_norm[l], c->rope, c->d_len, g.rms_eps, c->q, layer_k(c, l),
                                                 layer_v(c, l), c->slots, c->d_seq, c->ring != 0, st);
        }));
        TRY(timed(c, K_ATTN_DECODE, attn_decode_kernel_count(), st, [&] {
            return attn_decode_launch(c->q, layer_k(c, l), layer_v(c, l), B, g.n_q_heads, g.n_kv_heads, dh,
                                      c->slots, c->d_len, seq_map(c), c->dec_work, c->attn, c->d_err, c->len + 1, st);
        }));
        TRY(skinny(c, K_GEMM_O, c->tB_o[l], c->tX_attn, B, d, c->q_width, nullptr, s_o, st));
        TRY(timed(c, K_FINALIZE, 1, st, [&] {
            return finalize_residual_rmsnorm_launch(c->skinny_ws, s_o, d, c->x, c->post_norm[l], B, d, g.rms_eps, c->xn,
                                                    c->fin_part, c->fin_tick, st);
        }));
        TRY(skinny(c, K_GEMM_GATEUP, c->tB_gu[l], c->tX_xn, B, 2 * F, d, nullptr, s_gu, st));
        TRY(timed(c, K_FINALIZE, 1, st,
                  [&] { return finalize_swiglu_launch(c->skinny_ws, s_gu, 2 * F, c->h, B, F, st); }));
        TRY(skinny(c, K_GEMM_DOWN, c->tB_down[l], c->tX_h, B, d, F, nullptr, s_dn, st));
        const bool last = l == L - 1;
        TRY(timed(c, K_FINALIZE, 1, st, [&] {
            return finalize_residual_rmsnorm_launch(c->skinny_ws, s_dn, d, c->x, last ? c->final_norm : c->in_norm[l + 1],
                                                    B, d, g.rms_eps, last ? c->hn : c->xn, c->fin_part, c->fin_tick, st);
        }));
        if (l == c->tap_layer && c->tap_out)
            if (cudaMemcpyAsync(c->tap_out, c->x, (size_t)B * d * 2, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
                return QWEN3_E_CUDA;
    }
    TRY(skinny(c, K_GEMM_LMHEAD, c->tB_head, c->tX_hn, B, g.vocab, d, logits, 1, st));
    TRY(timed(c, K_LENGTH, 1, st, [&] { return add_len_launch(c->d_len, 1, st); }));
    return QWEN3_OK;
}

bool use_skinny_decode(const qwen3_ctx* c, int B) { return B <= kSkinnyRowsBox && c->cfg.hidden <= 4096; }

// One forward pass over M = B*T rows already gathered into c->x (T = 1 for decode).
int enqueue_forward(qwen3_ctx* c, const int32_t* ids, int B, int T, float* logits, int flags, bool decode,
                    cudaStream_t st) {
    const qwen3_config& g = c->cfg;
    if (decode && use_skinny_decode(c, B)) return enqueue_decode_skinny(c, ids, B, logits, st);
    const int M = B * T, d = g.hidden, dh = g.head_dim, F = g.intermediate;
    TRY(timed(c, K_EMBED, 1, st, [&] { return embed_launch(c->embed, g.vocab, d, ids, M, c->x, c->d_err, st); }));
    // Q [B*Hq][T][dh] store map for the fused QKV epilogue (used when T is a multiple of 128)
    CUtensorMap tq3;
    if (!encode_tmap_bf16_3d(&tq3, c->q, dh, T, (uint64_t)B * g.n_q_heads)) return QWEN3_E_CUDA;
    // o_proj and down_proj write the next RMSNorm's output too (all but the last layer's down_proj)
    const bool fuse = gemm_norm_preferred(M, d);
    for (int l = 0; l < g.n_layers; ++l) {
        if (l == c->tap_layer && c->tap_in)
            if (cudaMemcpyAsync(c->tap_in, c->x, (size_t)M * d * 2, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
                return QWEN3_E_CUDA;
        if (!fuse || l == 0)
            TRY(timed(c, K_RMSNORM, 1, st,
                      [&] { return rmsnorm_launch(c->x, c->in_norm[l], M, d, 1, 0, g.rms_eps, c->xn, st); }));
        {
            // fused: Q/K/V projection, q_norm/k_norm, RoPE, Q to attention layout, K/V into the cache
            GemmArgs a{M, c->qkv_n, d, EPI_QKV_ROPE, 1, nullptr, 0, nullptr, 0, c->d_err,
                       QkvRopeArgs{c->q_norm[l], c->k_norm[l], c->rope, c->d_len, c->q, layer_k(c, l), layer_v(c, l), T,
                                   g.n_q_heads, g.n_kv_heads, dh, c->slots, g.rms_eps, c->d_seq, c->ring != 0}};
            GemmMaps m;
            std::memset(&m, 0, sizeof(m));
            m.a = c->tA_xn;
            m.b = c->tB_qkv[l];
            m.c = tq3;
            m.r = c->tK3[l];
            m.v = c->tV3[l];
            TRY(timed(c, K_GEMM_QKV, 1, st, [&] { return gemm_launch(m, a, st); }));
        }
        if (decode) {
            TRY(timed(c, K_ATTN_DECODE, attn_decode_kernel_count(), st, [&] {
                return attn_decode_launch(c->q, layer_k(c, l), layer_v(c, l), B, g.n_q_heads, g.n_kv_heads, dh,
                                          c->slots, c->d_len, seq_map(c), c->dec_work, c->attn, c->d_err, c->len + 1,
                                          st);
            }));
        } else {
            int split = 0, chunks = 1;
            attn_prefill_split_plan(B, T, g.n_q_heads, g.n_kv_heads, c->len + T, &split, &chunks);
            if (attn_prefill_workspace(B, T, g.n_q_heads, g.n_kv_heads, dh, chunks) > c->attn_ws_bytes) {
                split = 0;
                chunks = 1;
            }
            TRY(timed(c, K_ATTN_PREFILL, 1, st, [&] {
                return attn_prefill_launch(c->q, layer_k(c, l), layer_v(c, l), B, T, g.n_q_heads, g.n_kv_heads, dh,
                                           c->slots, c->d_len, seq_map(c), c->attn, c->d_err, split, chunks,
                                           c->attn_ws, 0, c->len + T, st);
            }));
        }
        if (fuse) {
            TRY(gemm_norm(c, K_GEMM_O, c->tA_attn, c->tB_o[l], M, d, c->q_width, c->post_norm[l], st));
        } else {
            TRY(gemm(c, K_GEMM_O, c->tA_attn, c->tB_o[l], &c->tC_x, &c->tC_x, M, d, c->q_width, EPI_RESIDUAL, c->x, d,
                     c->x, d, st));
            TRY(timed(c, K_RMSNORM, 1, st,
                      [&] { return rmsnorm_launch(c->x, c->post_norm[l], M, d, 1, 0, g.rms_eps, c->xn, st); }));
        }
        TRY(gemm(c, K_GEMM_GATEUP, c->tA_xn, c->tB_gu[l], &c->tC_h, nullptr, M, 2 * F, d, EPI_SWIGLU, c->h, F,
                 nullptr, 0, st));
        if (fuse && l + 1 < g.n_layers) {
            TRY(gemm_norm(c, K_GEMM_DOWN, c->tA_h, c->tB_down[l], M, d, F, c->in_norm[l + 1], st));
        } else {
            TRY(gemm(c, K_GEMM_DOWN, c->tA_h, c->tB_down[l], &c->tC_x, &c->tC_x, M, d, F, EPI_RESIDUAL, c->x, d, c->x,
                     d, st));
        }
        if (l == c->tap_layer && c->tap_out)
            if (cudaMemcpyAsync(c->tap_out, c->x, (size_t)M * d * 2, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
                return QWEN3_E_CUDA;
    }
    const bool all_rows = decode || (flags & QWEN3_ALL_ROWS);
    const int rows = all_rows ? M : B;
    TRY(timed(c, K_RMSNORM, 1, st, [&] {
        return all_rows ? rmsnorm_launch(c->x, c->final_norm, rows, d, 1, 0, g.rms_eps, c->hn, st)
                        : rmsnorm_launch(c->x, c->final_norm, rows, d, T, T - 1, g.rms_eps, c->hn, st);
    }));
    if (rows <= kSkinnyRowsBox) {  // a few rows: stream the vocabulary matrix through the weight-streaming GEMM
        TRY(skinny(c, K_GEMM_LMHEAD, c->tB_head, c->tX_hn, rows, g.vocab, d, logits, 1, st));
        TRY(timed(c, K_LENGTH, 1, st, [&] { return add_len_launch(c->d_len, T, st); }));
        return QWEN3_OK;
    }
    CUtensorMap t_logits;
    if (!encode_tmap_out(&t_logits, logits, true, g.vocab, rows, g.vocab)) return QWEN3_E_CUDA;
    TRY(gemm(c, K_GEMM_LMHEAD, c->tA_hn, c->tB_head, &t_logits, nullptr, rows, g.vocab, d, EPI_F32, logits, g.vocab,
             nullptr, 0, st));
    TRY(timed(c, K_LENGTH, 1, st, [&] { return add_len_launch(c->d_len, T, st); }));
    return QWEN3_OK;
}

// Enqueue one forward pass, replaying a captured CUDA graph of it when the same call was made before
// (the whole pass is then one launch for the host). Timing, the debug tap and a caller's stream that is
// itself being captured run it eagerly.
int run_forward(qwen3_ctx* c, const int32_t* ids, int B, int T, float* logits, int flags, bool decode,
                cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return QWEN3_E_CUDA;
    // the caller's own capture records the launches themselves
    if (c->timing || c->tap_layer >= 0 || cs != cudaStreamCaptureStatusNone)
        return enqueue_forward(c, ids, B, T, logits, flags, decode, st);
    const int len = decode ? -attn_decode_chunks(c->len + 1, c->slots, c->window, c->ring) : c->len;
    ForwardGraph* gph = nullptr;
    for (auto& x : c->graphs)
        if (x.B == B && x.T == T && x.flags == flags && x.decode == (int)decode && x.len == len && x.ids == ids &&
            x.logits == logits)
            gph = &x;
    if (!gph) {
        cudaGraph_t graph = nullptr;
        cudaGraphExec_t exec = nullptr;
        if (cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return QWEN3_E_CUDA;
        const int rc = enqueue_forward(c, ids, B, T, logits, flags, decode, c->cap_stream);
        cudaError_t e = cudaStreamEndCapture(c->cap_stream, &graph);
        if (rc != QWEN3_OK) {
            if (graph) cudaGraphDestroy(graph);
            return rc;
        }
        if (e != cudaSuccess) return QWEN3_E_CUDA;
        e = cudaGraphInstantiate(&exec, graph, 0);
        cudaGraphDestroy(graph);
        if (e != cudaSuccess) return QWEN3_E_CUDA;
        if (c->graphs.size() >= kMaxGraphs) {
            cudaGraphExecDestroy(c->graphs.front().exec);
            c->graphs.erase(c->graphs.begin());
        }
        c->graphs.push_back({B, T, flags, (int)decode, len, ids, logits, exec});
        gph = &c->graphs.back();
    }
    return cudaGraphLaunch(gph->exec, st) == cudaSuccess ? QWEN3_OK : QWEN3_E_CUDA;
}

int check_call(qwen3_ctx* c, int B, int T) {
    if (B < 1 || T < 1) return QWEN3_E_ARG;
    if (B > c->max_batch || (long long)B * T > c->max_tokens) return QWEN3_E_BATCH;
    if (c->len > 0 && B != c->batch) return QWEN3_E_BATCH;
    if ((long long)c->len + T > c->capacity) return QWEN3_E_OVERFLOW;
    // a rolling buffer holds the window plus one call's tokens
    if (c->ring && T > c->ring - c->window + 1) return QWEN3_E_BATCH;
    return QWEN3_OK;
}

template <typename T>
cudaError_t dmalloc(T** p, size_t elems) {
    *p = nullptr;
    if (elems == 0) elems = 1;
    return cudaMalloc(reinterpret_cast<void**>(p), elems * sizeof(T));
}

void release(qwen3_ctx* c) {
    if (!c) return;
    for (auto& gph : c->graphs) cudaGraphExecDestroy(gph.exec);
    for (auto& t : c->timed) {
        cudaEventDestroy(t.start);
        cudaEventDestroy(t.stop);
    }
    for (auto e : c->free_events) cudaEventDestroy(e);
    if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
    void* bufs[] = {c->wqkv, c->wgu,      c->kcache, c->vcache, c->rope,      c->x,           c->xn,
                    c->q,    c->attn,     c->h,      c->hn,     c->dec_work,  c->attn_ws,     c->skinny_ws, c->d_len,
                    c->d_err, c->d_ids_buf, c->d_logits_buf, c->d_seq, c->gen_logits, c->gen_done, c->gen_next,
                    c->gen_alive, c->gen_work, c->fin_part, c->fin_tick, c->norm_part, c->norm_count};
    for (void* p : bufs)
        if (p) cudaFree(p);
    if (c->h_alive) cudaFreeHost(c->h_alive);
    delete c;
}

// Replace the device copy of the sequence layout (values travel inside the update launches; nothing
// is enqueued when the layout does not change).
int write_seq(qwen3_ctx* c, const std::vector<int>& v, cudaStream_t st) {
    if (v == c->h_seq) return QWEN3_OK;
    if (set_seq_launch(c->d_seq, v.data(), (int)v.size(), st) != cudaSuccess) return QWEN3_E_CUDA;
    c->h_seq = v;
    return QWEN3_OK;
}

// Buffers of the greedy generation loop, allocated on first use.
int ensure_generation_buffers(qwen3_ctx* c) {
    if (c->gen_logits) return QWEN3_OK;
    const size_t mb = (size_t)c->max_batch;
    if (dmalloc(&c->gen_logits, mb * c->cfg.vocab) != cudaSuccess || dmalloc(&c->gen_done, mb) != cudaSuccess ||
        dmalloc(&c->gen_next, mb) != cudaSuccess || dmalloc(&c->gen_alive, 1) != cudaSuccess ||
        dmalloc(&c->gen_work, greedy_workspace_ints((int)mb)) != cudaSuccess ||
        cudaMemset(c->gen_work, 0, greedy_workspace_ints((int)mb) * sizeof(int)) != cudaSuccess ||
        cudaMallocHost(reinterpret_cast<void**>(&c->h_alive), sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return QWEN3_E_CUDA;
    }
    return QWEN3_OK;
}

}  // namespace

extern "C" {

const char* qwen3_strerror(int code) {
    switch (code) {
        case QWEN3_OK: return "ok";
        case QWEN3_E_CONFIG: return "invalid or unsupported model configuration";
        case QWEN3_E_CAPACITY: return "requested cache exceeds the context limit";
        case QWEN3_E_OVERFLOW: return "sequence exceeds the cache capacity";
        case QWEN3_E_BATCH: return "batch or token count does not fit the context";
        case QWEN3_E_ARG: return "invalid argument";
        case QWEN3_E_CUDA: return "CUDA error";
        case QWEN3_E_TOKEN: return "token id out of range";
        case QWEN3_E_TIMEOUT: return "a kernel wait timed out";
        case QWEN3_E_DEVICE: return "device is not an sm_103 GPU";
    }
    return "unknown error";
}

int qwen3_validate_config(const qwen3_config* g) {
    if (!g) return QWEN3_E_ARG;
    if (g->n_layers < 1 || g->hidden < 64 || g->n_q_heads < 1 || g->n_kv_heads < 1 || g->intermediate < 128 ||
        g->vocab < 8 || g->max_positions < 1)
        return QWEN3_E_CONFIG;
    if (g->n_q_heads % g->n_kv_heads) return QWEN3_E_CONFIG;
    const int grp = g->n_q_heads / g->n_kv_heads;
    if (grp != 1 && grp != 2 && grp != 4 && grp != 8) return QWEN3_E_CONFIG;
    if (g->head_dim != 64 && g->head_dim != 128) return QWEN3_E_CONFIG;
    if (g->hidden % 64 || g->intermediate % 128 || g->vocab % 8 || g->hidden > 8192) return QWEN3_E_CONFIG;
    if (!(g->rms_eps > 0.f) || !(g->rope_theta > 1.f)) return QWEN3_E_CONFIG;
    if (g->sliding_window < 0 || (g->rolling_cache != 0 && g->rolling_cache != 1)) return QWEN3_E_CONFIG;
    if (g->rolling_cache && g->sliding_window < 1) return QWEN3_E_CONFIG;
    return QWEN3_OK;
}

int qwen3_init(const qwen3_config* g, const qwen3_weights* w, int max_batch, int capacity, int max_tokens,
               void* stream, qwen3_ctx** out) {
    if (!g || !w || !out) return QWEN3_E_ARG;
    *out = nullptr;
    TRY(qwen3_validate_config(g));
    if (max_batch < 1 || capacity < 1 || max_tokens < 0) return QWEN3_E_ARG;
    if (capacity > g->max_positions) return QWEN3_E_CAPACITY;
    if (!w->embed || !w->final_norm || (!g->tie_embeddings && !w->lm_head)) return QWEN3_E_ARG;
    const void* const* lists[] = {w->in_norm, w->q_proj, w->k_proj,    w->v_proj,  w->o_proj,   w->q_norm,
                                  w->k_norm,  w->post_norm, w->gate_proj, w->up_proj, w->down_proj};
    for (auto lst : lists) {
        if (!lst) return QWEN3_E_ARG;
        for (int l = 0; l < g->n_layers; ++l)
            if (!lst[l] || !is_aligned(lst[l], 16)) return QWEN3_E_ARG;
    }
    if (!device_is_sm103()) return QWEN3_E_DEVICE;
    if (prepare_kernels() != cudaSuccess) return QWEN3_E_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    qwen3_ctx* c = new (std::nothrow) qwen3_ctx();
    if (!c) return QWEN3_E_CUDA;
    c->cfg = *g;
    c->max_batch = max_batch;
    c->capacity = capacity;
    const long long mt = max_tokens > 0 ? (long long)max_tokens : (long long)max_batch * capacity;
    if (mt > (1ll << 30)) {
        delete c;
        return QWEN3_E_ARG;
    }
    c->max_tokens = (int)mt;
    c->window = g->sliding_window;
    if (g->rolling_cache) {
        // ring of W + (one sequence's share of a call) - 1 slots, a multiple of 256: no token of a call
        // overwrites a key that another token of the same call still sees (longer calls are refused)
        const long long chunk = std::min<long long>((mt + max_batch - 1) / max_batch, capacity);
        const long long need = (long long)g->sliding_window + chunk - 1;
        c->ring = (int)((need + 255) / 256 * 256);
        c->slots = c->ring;
    } else {
        c->slots = capacity;
    }
    const int L = g->n_layers, d = g->hidden, dh = g->head_dim, F = g->intermediate, V = g->vocab;
    c->q_width = g->n_q_heads * dh;
    c->qkv_n = (g->n_q_heads + 2 * g->n_kv_heads) * dh;
    const int kvw = g->n_kv_heads * dh;
    c->embed = static_cast<const bf16*>(w->embed);
    c->head = static_cast<const bf16*>(g->tie_embeddings ? w->embed : w->lm_head);
    c->final_norm = static_cast<const bf16*>(w->final_norm);
    for (int l = 0; l < L; ++l) {
        c->in_norm.push_back(static_cast<const bf16*>(w->in_norm[l]));
        c->q_norm.push_back(static_cast<const bf16*>(w->q_norm[l]));
        c->k_norm.push_back(static_cast<const bf16*>(w->k_norm[l]));
        c->post_norm.push_back(static_cast<const bf16*>(w->post_norm[l]));
        c->o_proj.push_back(static_cast<const bf16*>(w->o_proj[l]));
        c->down_proj.push_back(static_cast<const bf16*>(w->down_proj[l]));
    }
    c->layer_elems = (size_t)max_batch * g->n_kv_heads * c->slots * dh;
    const size_t rows = (size_t)c->max_tokens;
    // The A-operand buffers get at least one full 128-row tile so TMA boxes stay inside them.
    const size_t arows = rows < 128 ? 128 : rows;
    bool ok = dmalloc(&c->wqkv, (size_t)L * c->qkv_n * d) == cudaSuccess &&
              dmalloc(&c->wgu, (size_t)L * 2 * F * d) == cudaSuccess &&
              dmalloc(&c->kcache, (size_t)L * c->layer_elems) == cudaSuccess &&
              dmalloc(&c->vcache, (size_t)L * c->layer_elems) == cudaSuccess &&
              dmalloc(&c->rope, (size_t)capacity * dh) == cudaSuccess &&
              dmalloc(&c->x, rows * d) == cudaSuccess && dmalloc(&c->xn, arows * d) == cudaSuccess &&
              dmalloc(&c->q, rows * c->q_width) == cudaSuccess &&
              dmalloc(&c->attn, arows * c->q_width) == cudaSuccess && dmalloc(&c->h, arows * F) == cudaSuccess &&
              dmalloc(&c->hn, arows * d) == cudaSuccess &&
              dmalloc(&c->dec_work, attn_decode_workspace(max_batch, g->n_q_heads, dh, c->slots, c->window, c->ring) / 4) ==
                  cudaSuccess &&
              dmalloc(&c->d_seq, (size_t)kSeqMetaHead + max_batch) == cudaSuccess &&
              dmalloc(&c->d_len, 1) == cudaSuccess && dmalloc(&c->d_err, 1) == cudaSuccess &&
              dmalloc(&c->d_ids_buf, rows) == cudaSuccess &&
              dmalloc(&c->norm_part, gemm_norm_part_floats((int)rows)) == cudaSuccess &&
              dmalloc(&c->norm_count, gemm_norm_count_ints((int)rows)) == cudaSuccess;
    // decode split-K workspace: the largest [splits][64][N] fp32 set of slices over the four projections
    if (ok) {
        const long long need = std::max(
            std::max((long long)skinny_splits(c->qkv_n, d) * c->qkv_n, (long long)skinny_splits(d, c->q_width) * d),
            std::max((long long)skinny_splits(2 * F, d) * 2 * F, (long long)skinny_splits(d, F) * d));
        c->skinny_ld = need;
        ok = dmalloc(&c->skinny_ws, (size_t)kSkinnyRowsBox * need) == cudaSuccess &&
             dmalloc(&c->fin_part, (size_t)kSkinnyRowsBox * finalize_norm_chunks(d)) == cudaSuccess &&
             dmalloc(&c->fin_tick, (size_t)kSkinnyRowsBox) == cudaSuccess &&
             cudaMemsetAsync(c->fin_tick, 0, (size_t)kSkinnyRowsBox * sizeof(int), st) == cudaSuccess;
    }
    // split-attention workspace: sized for the largest split the planner can choose (work items up to
    // the SM count, up to 4 chunks each)
    if (ok) {
        const int nh = (g->n_q_heads / g->n_kv_heads) % 2 == 0 ? 2 : 1;
        c->attn_ws_bytes = ((size_t)device_sm_count() / 4 + 1) * 16 * nh * 128 * (dh + 4) * sizeof(float) + 4096;
        ok = dmalloc(&c->attn_ws, c->attn_ws_bytes / sizeof(float)) == cudaSuccess &&
             cudaMemsetAsync(c->attn_ws, 0, c->attn_ws_bytes, st) == cudaSuccess;
    }
    if (!ok) {
        cudaGetLastError();
        release(c);
        return QWEN3_E_CUDA;
    }
    // zero the cache and scratch so no stale bits are ever read, then pack the fused weights
    ok = cudaMemsetAsync(c->kcache, 0, (size_t)L * c->layer_elems * 2, st) == cudaSuccess &&
         cudaMemsetAsync(c->vcache, 0, (size_t)L * c->layer_elems * 2, st) == cudaSuccess &&
         cudaMemsetAsync(c->xn, 0, arows * d * 2, st) == cudaSuccess &&
         cudaMemsetAsync(c->attn, 0, arows * c->q_width * 2, st) == cudaSuccess &&
         cudaMemsetAsync(c->h, 0, arows * F * 2, st) == cudaSuccess &&
         cudaMemsetAsync(c->hn, 0, arows * d * 2, st) == cudaSuccess &&
         cudaMemsetAsync(c->d_len, 0, sizeof(int), st) == cudaSuccess &&
         cudaMemsetAsync(c->d_seq, 0, ((size_t)kSeqMetaHead + max_batch) * sizeof(int), st) == cudaSuccess &&
         cudaMemsetAsync(c->d_err, 0, sizeof(int), st) == cudaSuccess &&
         cudaMemsetAsync(c->norm_count, 0, gemm_norm_count_ints((int)rows) * sizeof(unsigned), st) == cudaSuccess;
    for (int l = 0; ok && l < L; ++l) {
        bf16* dst = c->wqkv + (size_t)l * c->qkv_n * d;
        ok = cudaMemcpyAsync(dst, w->q_proj[l], (size_t)c->q_width * d * 2, cudaMemcpyDeviceToDevice, st) ==
                 cudaSuccess &&
             cudaMemcpyAsync(dst + (size_t)c->q_width * d, w->k_proj[l], (size_t)kvw * d * 2,
                             cudaMemcpyDeviceToDevice, st) == cudaSuccess &&
             cudaMemcpyAsync(dst + (size_t)(c->q_width + kvw) * d, w->v_proj[l], (size_t)kvw * d * 2,
                             cudaMemcpyDeviceToDevice, st) == cudaSuccess &&
             pack_gate_up_launch(static_cast<const bf16*>(w->gate_proj[l]), static_cast<const bf16*>(w->up_proj[l]), F,
                                 d, c->wgu + (size_t)l * 2 * F * d, st) == cudaSuccess;
    }
    ok = ok && rope_table_launch(g->rope_theta, dh, capacity, c->rope, st) == cudaSuccess;
    // tensor maps
    ok = ok && encode_tmap_bf16_2d(&c->tA_xn, c->xn, d, arows, (uint64_t)d * 2, kGemmBK, kGemmBM) &&
         encode_tmap_bf16_2d(&c->tA_attn, c->attn, c->q_width, arows, (uint64_t)c->q_width * 2, kGemmBK, kGemmBM) &&
         encode_tmap_bf16_2d(&c->tA_h, c->h, F, arows, (uint64_t)F * 2, kGemmBK, kGemmBM) &&
         encode_tmap_bf16_2d(&c->tA_hn, c->hn, d, arows, (uint64_t)d * 2, kGemmBK, kGemmBM) &&
         encode_tmap_bf16_2d(&c->tB_head, c->head, d, V, (uint64_t)d * 2, kGemmBK, kGemmBoxN) &&
         encode_tmap_out(&c->tC_x, c->x, false, d, rows, d) && encode_tmap_out(&c->tC_h, c->h, false, F, arows, F) &&
         encode_tmap_out(&c->tC_xn, c->xn, false, d, arows, d) &&
         encode_skinny_x_map(&c->tX_xn, c->xn, arows, d) && encode_skinny_x_map(&c->tX_attn, c->attn, arows, c->q_width) &&
         encode_skinny_x_map(&c->tX_h, c->h, arows, F) && encode_skinny_x_map(&c->tX_hn, c->hn, arows, d);
    c->tK3.resize(L);
    c->tV3.resize(L);
    for (int l = 0; ok && l < L; ++l)
        ok = encode_tmap_bf16_3d(&c->tK3[l], c->kcache + (size_t)l * c->layer_elems, dh, c->slots,
                                 (uint64_t)max_batch * g->n_kv_heads) &&
             encode_tmap_bf16_3d(&c->tV3[l], c->vcache + (size_t)l * c->layer_elems, dh, c->slots,
                                 (uint64_t)max_batch * g->n_kv_heads);
    c->tB_qkv.resize(L);
    c->tB_o.resize(L);
    c->tB_gu.resize(L);
    c->tB_down.resize(L);
    for (int l = 0; ok && l < L; ++l) {
        ok = encode_tmap_bf16_2d(&c->tB_qkv[l], c->wqkv + (size_t)l * c->qkv_n * d, d, c->qkv_n, (uint64_t)d * 2,
                                 kGemmBK, kGemmBoxN) &&
             encode_tmap_bf16_2d(&c->tB_o[l], c->o_proj[l], c->q_width, d, (uint64_t)c->q_width * 2, kGemmBK, kGemmBoxN) &&
             encode_tmap_bf16_2d(&c->tB_gu[l], c->wgu + (size_t)l * 2 * F * d, d, 2 * F, (uint64_t)d * 2, kGemmBK,
                                 kGemmBoxN) &&
             encode_tmap_bf16_2d(&c->tB_down[l], c->down_proj[l], F, d, (uint64_t)F * 2, kGemmBK, kGemmBoxN);
    }
    ok = ok && cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking) == cudaSuccess;
    ok = ok && cudaStreamSynchronize(st) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        release(c);
        return QWEN3_E_CUDA;
    }
    c->h_seq.assign((size_t)kSeqMetaHead + max_batch, 0);
    *out = c;
    return QWEN3_OK;
}

int qwen3_prefill(qwen3_ctx* c, const int32_t* d_ids, int B, int T, float* d_logits, int flags, void* stream) {
    if (!c || !d_ids || !d_logits) return QWEN3_E_ARG;
    TRY(check_call(c, B, T));
    TRY(run_forward(c, d_ids, B, T, d_logits, flags, false, static_cast<cudaStream_t>(stream)));
    c->len += T;
    c->batch = B;
    return QWEN3_OK;
}

int qwen3_decode_step(qwen3_ctx* c, const int32_t* d_ids, int B, float* d_logits, void* stream) {
    if (!c || !d_ids || !d_logits) return QWEN3_E_ARG;
    TRY(check_call(c, B, 1));
    TRY(run_forward(c, d_ids, B, 1, d_logits, 0, true, static_cast<cudaStream_t>(stream)));
    c->len += 1;
    c->batch = B;
    return QWEN3_OK;
}

int qwen3_prefill_padded(qwen3_ctx* c, const int32_t* d_ids, const int32_t* h_real, int B, int T, float* d_logits,
                         int flags, void* stream) {
    if (!c || !d_ids || !h_real || !d_logits) return QWEN3_E_ARG;
    TRY(check_call(c, B, T));
    if (c->window > 0) return QWEN3_E_ARG;  // padding and sliding windows are not combined
    std::vector<int> v = c->h_seq;
    int any = 0;
    for (int b = 0; b < B; ++b) {
        if (h_real[b] < 1 || h_real[b] > T) return QWEN3_E_ARG;
        any |= T - h_real[b];
    }
    if (any && c->padded) return QWEN3_E_ARG;  // one padded block per fill of the cache
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (any) {
        v[0] = c->len;
        for (int b = 0; b < c->max_batch; ++b) v[kSeqMetaHead + b] = b < B ? T - h_real[b] : 0;
        TRY(write_seq(c, v, st));
        c->padded = true;
    }
    TRY(run_forward(c, d_ids, B, T, d_logits, flags, false, st));
    c->len += T;
    c->batch = B;
    return QWEN3_OK;
}

int qwen3_share_prefix(qwen3_ctx* c, int B, void* stream) {
    if (!c) return QWEN3_E_ARG;
    if (B < 1 || B > c->max_batch) return QWEN3_E_BATCH;
    if (c->batch != 1 || c->len < 1 || c->padded || c->window > 0 || c->h_seq[1] > 0) return QWEN3_E_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int psh = c->len / 128 * 128;  // whole 128-slot tiles are read from sequence 0 in place
    if (copy_prefix_slots_launch(c->kcache, c->vcache, c->layer_elems, c->cfg.n_layers, B, c->cfg.n_kv_heads, c->slots,
                                 c->cfg.head_dim, psh, c->len, st) != cudaSuccess)
        return QWEN3_E_CUDA;
    std::vector<int> v = c->h_seq;
    v[1] = psh;
    TRY(write_seq(c, v, st));
    c->batch = B;
    return QWEN3_OK;
}

int qwen3_generate(qwen3_ctx* c, const int32_t* d_ids, const int32_t* h_real, int B, int T, int max_new, int stop_id,
                   int32_t* d_out, int* h_steps, void* stream) {
    if (!c || !d_ids || !d_out || max_new < 1) return QWEN3_E_ARG;
    if (stop_id >= c->cfg.vocab) return QWEN3_E_ARG;
    if (c->len + T + max_new - 1 > c->capacity) return QWEN3_E_OVERFLOW;
    TRY(ensure_generation_buffers(c));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int V = c->cfg.vocab;
    if (h_real) {
        TRY(qwen3_prefill_padded(c, d_ids, h_real, B, T, c->gen_logits, 0, stream));
    } else {
        TRY(qwen3_prefill(c, d_ids, B, T, c->gen_logits, 0, stream));
    }
    if (cudaMemsetAsync(c->gen_done, 0, (size_t)B * sizeof(int), st) != cudaSuccess) return QWEN3_E_CUDA;
    int steps = 0;
    for (;;) {
        if (cudaMemsetAsync(c->gen_alive, 0, sizeof(int), st) != cudaSuccess) return QWEN3_E_CUDA;
        if (greedy_launch(c->gen_logits, V, B, V, stop_id, stop_id >= 0 ? c->gen_done : nullptr, c->gen_next, d_out,
                          max_new, steps, c->gen_alive, c->gen_work, st) != cudaSuccess)
            return QWEN3_E_CUDA;
        ++steps;
        if (steps == max_new) break;
        if (stop_id >= 0) {  // stop once every row has finished
            if (cudaMemcpyAsync(c->h_alive, c->gen_alive, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
                cudaStreamSynchronize(st) != cudaSuccess)
                return QWEN3_E_CUDA;
            if (*c->h_alive == 0) break;
        }
        TRY(qwen3_decode_step(c, c->gen_next, B, c->gen_logits, stream));
    }
    if (h_steps) *h_steps = steps;
    return QWEN3_OK;
}

size_t qwen3_greedy_workspace(int B) { return B < 1 ? 0 : greedy_workspace_ints(B) * sizeof(int); }

int qwen3_op_greedy(const float* logits, int64_t ld, int B, int V, int stop_id, int32_t* done, int32_t* next,
                    int32_t* work, void* stream) {
    if (!logits || !next || B < 0 || V < 4 || V % 4 || ld < V || ld % 4 || !is_aligned(logits, 16)) return QWEN3_E_ARG;
    if (stop_id >= V || (work && !is_aligned(work, 16))) return QWEN3_E_ARG;
    return greedy_launch(logits, ld, B, V, stop_id, stop_id >= 0 ? done : nullptr, next, nullptr, 0, 0, nullptr, work,
                         static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QWEN3_OK
               : QWEN3_E_CUDA;
}

int qwen3_prefill_host(qwen3_ctx* c, const int32_t* h_ids, int B, int T, float* h_logits, int flags, void* stream) {
    if (!c || !h_ids || !h_logits) return QWEN3_E_ARG;
    TRY(check_call(c, B, T));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t rows = (flags & QWEN3_ALL_ROWS) ? (size_t)B * T : (size_t)B;
    const size_t need = rows * c->cfg.vocab;
    if (need > c->logits_buf_elems) {
        if (c->d_logits_buf) cudaFree(c->d_logits_buf);
        c->d_logits_buf = nullptr;
        c->logits_buf_elems = 0;
        if (dmalloc(&c->d_logits_buf, need) != cudaSuccess) return QWEN3_E_CUDA;
        c->logits_buf_elems = need;
    }
    if (cudaMemcpyAsync(c->d_ids_buf, h_ids, (size_t)B * T * 4, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return QWEN3_E_CUDA;
    TRY(qwen3_prefill(c, c->d_ids_buf, B, T, c->d_logits_buf, flags, stream));
    if (cudaMemcpyAsync(h_logits, c->d_logits_buf, need * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return QWEN3_E_CUDA;
    return qwen3_get_error(c, stream);
}

int qwen3_length(const qwen3_ctx* c, int* length, int* batch) {
    if (!c) return QWEN3_E_ARG;
    if (length) *length = c->len;
    if (batch) *batch = c->batch;
    return QWEN3_OK;
}

int qwen3_set_length(qwen3_ctx* c, int length, int batch, void* stream) {
    if (!c || length < 0) return QWEN3_E_ARG;
    if (length > c->capacity) return QWEN3_E_OVERFLOW;
    if (batch < 0 || batch > c->max_batch) return QWEN3_E_BATCH;
    if (set_len_launch(c->d_len, length, static_cast<cudaStream_t>(stream)) != cudaSuccess) return QWEN3_E_CUDA;
    c->len = length;
    c->batch = batch;
    // the cache now holds plain equal-length sequences: no padding, no shared prefix
    TRY(write_seq(c, std::vector<int>(c->h_seq.size(), 0), static_cast<cudaStream_t>(stream)));
    c->padded = false;
    return QWEN3_OK;
}

int qwen3_kv_view(qwen3_ctx* c, int layer, void** d_k, void** d_v, int64_t dims[4]) {
    if (!c || layer < 0 || layer >= c->cfg.n_layers) return QWEN3_E_ARG;
    if (d_k) *d_k = layer_k(c, layer);
    if (d_v) *d_v = layer_v(c, layer);
    if (dims) {
        dims[0] = c->max_batch;
        dims[1] = c->cfg.n_kv_heads;
        dims[2] = c->slots;
        dims[3] = c->cfg.head_dim;
    }
    return QWEN3_OK;
}

int qwen3_set_tap(qwen3_ctx* c, int layer, void* d_in, void* d_out) {
    if (!c || layer >= c->cfg.n_layers) return QWEN3_E_ARG;
    c->tap_layer = layer < 0 ? -1 : layer;
    c->tap_in = layer < 0 ? nullptr : d_in;
    c->tap_out = layer < 0 ? nullptr : d_out;
    return QWEN3_OK;
}

int qwen3_get_error(qwen3_ctx* c, void* stream) {
    if (!c) return QWEN3_E_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return QWEN3_E_CUDA;
    int flags = 0;
    if (cudaMemcpy(&flags, c->d_err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return QWEN3_E_CUDA;
    if (flags && cudaMemset(c->d_err, 0, sizeof(int)) != cudaSuccess) return QWEN3_E_CUDA;
    if (flags & ERR_TIMEOUT) return QWEN3_E_TIMEOUT;
    if (flags & ERR_TOKEN) return QWEN3_E_TOKEN;
    return QWEN3_OK;
}

int qwen3_set_timing(qwen3_ctx* c, int enable) {
    if (!c) return QWEN3_E_ARG;
    c->timing = enable != 0;
    return QWEN3_OK;
}

int qwen3_kernel_times(qwen3_ctx* c, double* total_ms, int64_t* launches, int* n) {
    if (!c || !n) return QWEN3_E_ARG;
    const int cap = *n;
    *n = K_NUM_CLASSES;
    for (int i = 0; i < cap && i < K_NUM_CLASSES; ++i) {
        if (total_ms) total_ms[i] = 0;
        if (launches) launches[i] = 0;
    }
    if (c->have_timed && cudaStreamSynchronize(c->last_timed) != cudaSuccess) return QWEN3_E_CUDA;
    c->have_timed = false;
    bool bad = false;
    for (auto& t : c->timed) {
        float ms = 0.f;
        bad = bad || cudaEventElapsedTime(&ms, t.start, t.stop) != cudaSuccess;
        if (t.cls < cap) {
            if (total_ms) total_ms[t.cls] += ms;
            if (launches) launches[t.cls] += t.launches;
        }
        c->free_events.push_back(t.start);
        c->free_events.push_back(t.stop);
    }
    c->timed.clear();
    return bad ? QWEN3_E_CUDA : QWEN3_OK;
}

const char* qwen3_kernel_class_name(int i) { return (i >= 0 && i < K_NUM_CLASSES) ? kClassNames[i] : nullptr; }

int qwen3_launch_count(const qwen3_ctx* c, int B, int T, int flags, int decode) {
    (void)flags;
    if (!c) return -1;
    if (decode && use_skinny_decode(c, B)) return 2 + c->cfg.n_layers * (8 + attn_decode_kernel_count()) + 2;
    const int per_layer = 6 + (decode ? attn_decode_kernel_count() : 1);
    if (gemm_norm_preferred(B * T, c->cfg.hidden))  // one RMSNorm launch per forward instead of two per layer
        return 1 + c->cfg.n_layers * (per_layer - 2) + 1 + 3;
    return 1 + c->cfg.n_layers * per_layer + 3;
}

void qwen3_free(qwen3_ctx* c) {
    if (!c) return;
    cudaDeviceSynchronize();
    release(c);
}

// ------------------------------------------------------------------------------ single operations

int qwen3_op_embed(const void* E, int V, int d, const int32_t* ids, int M, void* out, int* err, void* stream) {
    if (!E || !ids || !out || V < 1 || d < 8 || d % 8 || M < 0) return QWEN3_E_ARG;
    return embed_launch(static_cast<const bf16*>(E), V, d, ids, M, static_cast<bf16*>(out), err,
                        static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QWEN3_OK
               : QWEN3_E_CUDA;
}

int qwen3_op_rmsnorm(const void* x, const void* gamma, int rows, int n, int in_stride, int in_offset, float eps,
                     void* y, void* stream) {
    if (!x || !gamma || !y || rows < 0 || n < 8 || n % 8 || n > 8192 || in_stride < 1 || in_offset < 0)
        return QWEN3_E_ARG;
    return rmsnorm_launch(static_cast<const bf16*>(x), static_cast<const bf16*>(gamma), rows, n, in_stride, in_offset,
                          eps, static_cast<bf16*>(y), static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QWEN3_OK
               : QWEN3_E_CUDA;
}

int qwen3_op_gemm(const void* A, const void* B, int M, int N, int K, int epi, void* C, int ldc, const void* R, int ldr,
                  int* err, void* stream) {
    if (!A || !B || !C || M < 0 || N < 1 || K < 8 || K % 8 || epi < 0 || epi > 3) return QWEN3_E_ARG;
    if (epi == EPI_SWIGLU && N % 256) return QWEN3_E_ARG;
    if (epi == EPI_RESIDUAL && !R) return QWEN3_E_ARG;
    if (ldc < (epi == EPI_SWIGLU ? N / 2 : N) || ldc % (epi == EPI_F32 ? 4 : 8)) return QWEN3_E_ARG;
    if (epi == EPI_RESIDUAL && (ldr < N || ldr % 8)) return QWEN3_E_ARG;
    if (!is_aligned(A, 16) || !is_aligned(B, 16) || !is_aligned(C, 16) || (R && !is_aligned(R, 16)))
        return QWEN3_E_ARG;
    if (M == 0) return QWEN3_OK;
    if (prepare_kernels() != cudaSuccess) return QWEN3_E_CUDA;
    GemmMaps m;
    std::memset(&m, 0, sizeof(m));
    if (!encode_gemm_maps(&m.a, &m.b, A, (uint64_t)M, B, (uint64_t)N, (uint64_t)K)) return QWEN3_E_CUDA;
    const uint64_t out_cols = epi == EPI_SWIGLU ? (uint64_t)N / 2 : (uint64_t)N;
    if (!encode_tmap_out(&m.c, C, epi == EPI_F32, out_cols, (uint64_t)M, (uint64_t)ldc)) return QWEN3_E_CUDA;
    if (epi == EPI_RESIDUAL && !encode_tmap_out(&m.r, R, false, (uint64_t)N, (uint64_t)M, (uint64_t)ldr))
        return QWEN3_E_CUDA;
    GemmArgs a{M, N, K, epi, 0, C, ldc, static_cast<const bf16*>(R), ldr, err, {}};
    return gemm_launch(m, a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? QWEN3_OK : QWEN3_E_CUDA;
}

int qwen3_gemm_norm_supported(int M, int N) { return (M > 0 && N >= 128 && gemm_norm_fusable(M, N)) ? 1 : 0; }

size_t qwen3_gemm_norm_part_floats(int M) { return M > 0 ? gemm_norm_part_floats(M) + gemm_norm_count_ints(M) : 0; }

int qwen3_op_gemm_residual_norm(const void* A, const void* B, int M, int N, int K, void* X, const void* gamma, float eps,
                                void* Y, float* part, int* err, void* stream) {
    if (!A || !B || !X || !gamma || !Y || !part || M < 0 || N < 1 || K < 8 || K % 8) return QWEN3_E_ARG;
    if (!is_aligned(A, 16) || !is_aligned(B, 16) || !is_aligned(X, 16) || !is_aligned(Y, 16) || !is_aligned(gamma, 16))
        return QWEN3_E_ARG;
    if (M == 0) return QWEN3_OK;
    if (!qwen3_gemm_norm_supported(M, N)) return QWEN3_E_ARG;
    if (prepare_kernels() != cudaSuccess) return QWEN3_E_CUDA;
    GemmMaps m;
    std::memset(&m, 0, sizeof(m));
    if (!encode_gemm_maps(&m.a, &m.b, A, (uint64_t)M, B, (uint64_t)N, (uint64_t)K) ||
        !encode_tmap_out(&m.c, X, false, (uint64_t)N, (uint64_t)M, (uint64_t)N) ||
        !encode_tmap_out(&m.r, X, false, (uint64_t)N, (uint64_t)M, (uint64_t)N) ||
        !encode_tmap_out(&m.v, Y, false, (uint64_t)N, (uint64_t)M, (uint64_t)N))
        return QWEN3_E_CUDA;
    GemmArgs a{M, N, K, EPI_RESIDUAL_NORM, 0, X, N, static_cast<const bf16*>(X), N, err, {},
               NormArgs{static_cast<const bf16*>(gamma), eps, part,
                        reinterpret_cast<unsigned*>(part + gemm_norm_part_floats(M))}};
    return gemm_launch(m, a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? QWEN3_OK : QWEN3_E_CUDA;
}

int qwen3_gemm_skinny_splits(int N, int K) { return (N < 1 || K < 8) ? 1 : skinny_splits(N, K); }

int qwen3_op_gemm_skinny(const void* A, const void* B, int M, int N, int K, int splits, float* slices, float* out,
                         int* err, void* stream) {
    if (!A || !B || M < 1 || M > kSkinnyRowsBox || N < 1 || K < 8 || K % 8 || splits < 1 || splits > 64) return QWEN3_E_ARG;
    if ((splits == 1 && !out) || (splits > 1 && !slices)) return QWEN3_E_ARG;
    if (!is_aligned(A, 16) || !is_aligned(B, 16)) return QWEN3_E_ARG;
    const int k_blocks = (K + kGemmBK - 1) / kGemmBK;
    if ((k_blocks + splits - 1) / splits * (splits - 1) >= k_blocks) return QWEN3_E_ARG;  // no empty split
    if (prepare_kernels() != cudaSuccess) return QWEN3_E_CUDA;
    CUtensorMap tw, tx;
    if (!encode_tmap_bf16_2d(&tw, B, K, N, (uint64_t)K * 2, kGemmBK, kGemmBoxN) ||
        !encode_skinny_x_map(&tx, A, (uint64_t)M, (uint64_t)K))
        return QWEN3_E_CUDA;
    SkinnyArgs a{M, N, K, splits, slices, N, splits == 1 ? out : nullptr, N, err, 0};
    return gemm_skinny_launch(tw, tx, a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? QWEN3_OK : QWEN3_E_CUDA;
}

int qwen3_op_pack_gate_up(const void* gate, const void* up, int F, int d, void* out, void* stream) {
    if (!gate || !up || !out || F < 128 || F % 128 || d < 8) return QWEN3_E_ARG;
    return pack_gate_up_launch(static_cast<const bf16*>(gate), static_cast<const bf16*>(up), F, d,
                               static_cast<bf16*>(out), static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QWEN3_OK
               : QWEN3_E_CUDA;
}

int qwen3_op_rope_table(float theta, int dh, int n_pos, void* table, void* stream) {
    if (!table || (dh != 64 && dh != 128) || n_pos < 0) return QWEN3_E_ARG;
    return rope_table_launch(theta, dh, n_pos, static_cast<bf16*>(table), static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? QWEN3_OK
               : QWEN3_E_CUDA;
}

int qwen3_op_qknorm_rope_append(const void* qkv, int B, int T, int Hq, int Hkv, int dh, const void* qg, const void* kg,
                                const void* table, const int* len0, float eps, void* q_out, void* kc, void* vc, int cap,
                                void* stream) {
    if (!qkv || !qg || !kg || !table || !len0 || !q_out || !kc || !vc) return QWEN3_E_ARG;
    if (B < 0 || T < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv || (dh != 64 && dh != 128) || cap < 1) return QWEN3_E_ARG;
    return qknorm_rope_append_launch(static_cast<const bf16*>(qkv), B, T, Hq, Hkv, dh, static_cast<const bf16*>(qg),
                                     static_cast<const bf16*>(kg), static_cast<const bf16*>(table), len0, eps,
                                     static_cast<bf16*>(q_out), static_cast<bf16*>(kc), static_cast<bf16*>(vc), cap,
                                     static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QWEN3_OK
               : QWEN3_E_CUDA;
}

size_t qwen3_attention_prefill_workspace(int B, int T, int Hq, int Hkv, int dh, int kv_chunks) {
    if (B < 1 || T < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv) return 0;
    return attn_prefill_workspace(B, T, Hq, Hkv, dh, kv_chunks);
}

int qwen3_op_attention_prefill(const void* q, const void* kc, const void* vc, int B, int T, int Hq, int Hkv, int dh,
                               int cap, const int* len0, const int* seq_meta, int window, int ring, int heads_per_cta,
                               int kv_split, int kv_chunks, void* work, void* out, int* err, void* stream) {
    if (!q || !kc || !vc || !len0 || !out || B < 0 || T < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv ||
        (dh != 64 && dh != 128) || cap < 1 || kv_split < 0 || kv_chunks > 64 || (kv_split > 0 && !work))
        return QWEN3_E_ARG;
    if (window < 0 || (ring && (ring != cap || ring % 256 || window < 1))) return QWEN3_E_ARG;
    if (heads_per_cta < 0 || heads_per_cta > 2 || (heads_per_cta == 2 && (Hq / Hkv) % 2)) return QWEN3_E_ARG;
    if (prepare_kernels() != cudaSuccess) return QWEN3_E_CUDA;
    return attn_prefill_launch(static_cast<const bf16*>(q), static_cast<const bf16*>(kc), static_cast<const bf16*>(vc),
                               B, T, Hq, Hkv, dh, cap, len0, SeqMap{seq_meta, window, ring}, static_cast<bf16*>(out),
                               err, kv_split,
                               kv_chunks < 1 ? 1 : kv_chunks, static_cast<float*>(work), heads_per_cta, T,
                               static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QWEN3_OK
               : QWEN3_E_CUDA;
}

size_t qwen3_attention_decode_workspace(int B, int Hq, int dh, int cap, int window, int ring) {
    if (B < 1 || Hq < 1 || cap < 1 || window < 0 || ring < 0) return 0;
    return attn_decode_workspace(B, Hq, dh, cap, window, ring);
}

int qwen3_op_attention_decode(const void* q, const void* kc, const void* vc, int B, int Hq, int Hkv, int dh, int cap,
                              const int* len0, const int* seq_meta, int window, int ring, void* work, void* out,
                              int* err, void* stream) {
    if (!q || !kc || !vc || !len0 || !work || !out || B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv ||
        (dh != 64 && dh != 128) || cap < 1)
        return QWEN3_E_ARG;
    if (window < 0 || (ring && (ring != cap || ring % 256 || window < 1))) return QWEN3_E_ARG;
    const int grp = Hq / Hkv;
    if (grp != 1 && grp != 2 && grp != 4 && grp != 8) return QWEN3_E_ARG;
    if (prepare_kernels() != cudaSuccess) return QWEN3_E_CUDA;
    return attn_decode_launch(static_cast<const bf16*>(q), static_cast<const bf16*>(kc), static_cast<const bf16*>(vc), B,
                              Hq, Hkv, dh, cap, len0, SeqMap{seq_meta, window, ring}, static_cast<float*>(work),
                              static_cast<bf16*>(out), err, 0, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QWEN3_OK
               : QWEN3_E_CUDA;
}

int qwen3_op_attention_decode_noalloc(const void* q, const void* kc, const void* vc, int B, int Hq, int Hkv, int dh,
                                      int cap, const int* len0, void* out, int* err, void* stream) {
    if (!q || !kc || !vc || !len0 || !out || B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv || (dh != 64 && dh != 128) ||
        cap < 1)
        return QWEN3_E_ARG;
    const int grp = Hq / Hkv;
    if (grp != 1 && grp != 2 && grp != 4 && grp != 8) return QWEN3_E_ARG;
    if (attn_decode_workspace(B, Hq, dh, cap, 0, 0) > attn_decode_noalloc_max_bytes()) return QWEN3_E_ARG;
    if (prepare_kernels() != cudaSuccess) return QWEN3_E_CUDA;
    float* scratch = nullptr;
    if (attn_decode_noalloc_scratch(&scratch) != cudaSuccess) return QWEN3_E_CUDA;
    return attn_decode_launch(static_cast<const bf16*>(q), static_cast<const bf16*>(kc), static_cast<const bf16*>(vc), B,
                              Hq, Hkv, dh, cap, len0, SeqMap{}, scratch, static_cast<bf16*>(out), err, 0,
                              static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? QWEN3_OK
               : QWEN3_E_CUDA;
}

}  // extern "C"
