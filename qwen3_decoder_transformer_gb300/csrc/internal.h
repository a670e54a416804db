// Internal launch interface between the kernel files and the runtime (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace q3 {

// Launch with programmatic stream serialization, so the kernel's prologue can overlap the tail of the
// previous kernel on the stream; every kernel of this library calls pdl_wait() before touching memory
// that earlier kernels produce or read.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Device error-flag bits (one int per context, read by qwen3_get_error).
enum : int { ERR_TOKEN = 1, ERR_TIMEOUT = 2 };

enum Epilogue : int { EPI_BF16 = 0, EPI_SWIGLU = 1, EPI_RESIDUAL = 2, EPI_F32 = 3, EPI_QKV_ROPE = 4, EPI_RESIDUAL_NORM = 5 };

// ---------------------------------------------------------------- host utilities (gemm.cu)
int device_sm_count();
bool device_is_sm103();
// Encode a 2-D bf16 tensor map over a row-major [outer, inner] matrix with the 128-byte swizzle.
bool encode_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                         uint32_t box_inner, uint32_t box_outer);

// ---------------------------------------------------------------- GEMM (gemm.cu)
// Extra operands of EPI_QKV_ROPE: the accumulator row of a QKV tile is one token's q/k/v head
// vectors; the epilogue applies q_norm/k_norm and RoPE and writes Q [B, Hq, T, dh] and the cache.
struct QkvRopeArgs {
    const __nv_bfloat16 *q_gamma, *k_gamma, *table;  // table [positions][dh]: cos then sin per position
    const int* len0;                                  // device cache length (first new slot)
    __nv_bfloat16 *q_out, *k_cache, *v_cache;        // caches [B][Hkv][cap][dh]
    int T, Hq, Hkv, dh, cap;                          // cap: physical slots per (sequence, kv head)
    float eps;
    const int* meta;  // sequence layout (SeqMap::meta), or null
    int rolling;      // nonzero: slot s is stored at s mod cap (cap a multiple of 256)
};
// Layout of each sequence's cache, read by the kernels that place or read keys:
//   meta (device ints, null for plain equal-length sequences): meta[0] = ps, the first padding slot;
//   meta[1] = psh, slots below it are read from sequence 0's cache (a multiple of 128, shared
//   prefix); meta[2 + b] = the number of padding slots of sequence b, [ps, ps + pad_b).
//   Slot s of sequence b holds position s below ps, max(ps - 1, 0) in the padding, s - pad_b after it.
//   A query in slot q sees key slot k iff (k <= q, k is not padding and, with a window W > 0,
//   q - k < W) or k == q.
//   ring: 0 = slot s is stored at s; otherwise at s mod ring (rolling buffer).
struct SeqMap {
    const int* meta;
    int window;
    int ring;
};
constexpr int kSeqMetaHead = 2;
constexpr int kSeqChunk = 1000;  // ints per set_seq launch (carried as a kernel parameter)
cudaError_t set_seq_launch(int* dst, const int* vals, int n, cudaStream_t st);
// EPI_RESIDUAL_NORM: the residual epilogue followed by the next RMSNorm of the updated rows,
// Y = bf16(gamma * bf16(X * rsqrt(mean(X^2) + eps))) with X the new residual stream. The N / BN column
// tiles of a row block (at most 8) run at the same time on different CTAs of one cooperative launch and
// exchange per-row partial sums of squares through part ([row blocks][8 tiles][2 halves][128] floats), meeting on
// count ([row blocks][2]: arrivals, departures; zero before the first launch, left zero by each).
struct NormArgs {
    const __nv_bfloat16* gamma;
    float eps;
    float* part;
    unsigned* count;
};
struct GemmArgs {
    int M, N, K;
    int epi;
    int b_independent;  // nonzero: B is not written by the previous kernel on the stream (model weights)
    void* C;
    long long ldc;
    const __nv_bfloat16* R;
    long long ldr;
    int* err;
    QkvRopeArgs qkv;
    NormArgs norm;
};
// Whether EPI_RESIDUAL_NORM can run for an [M, N] output (N a multiple of the tile width, at most 8
// tiles); the sizes of NormArgs::part (floats) and NormArgs::count (ints) for up to M rows.
bool gemm_norm_fusable(int M, int N);
bool gemm_norm_preferred(int M, int N);  // fusable and expected to beat GEMM + separate RMSNorm
size_t gemm_norm_part_floats(int M);
size_t gemm_norm_count_ints(int M);
// Tile rows of A, TMA box rows of B (a 256-wide tile loads two boxes), K per stage.
constexpr int kGemmBM = 128, kGemmBoxN = 128, kGemmBK = 64;
// A: [rows >= M, K] activations; B: [N, K] weights. Both maps are built with encode_gemm_maps.
bool encode_gemm_maps(CUtensorMap* ta, CUtensorMap* tb, const void* A, uint64_t a_rows, const void* B, uint64_t N,
                      uint64_t K);
// Output / residual map for the staged epilogues: a [rows, cols] matrix with row stride ld elements,
// boxes of 128 rows x 128 bytes (64 bf16 or 32 fp32 columns).
bool encode_tmap_out(CUtensorMap* map, const void* base, bool f32, uint64_t cols, uint64_t rows, uint64_t ld);
// The tensor maps of one GEMM launch: A, B, the output C (staged epilogues) and the residual R. The
// fused QKV epilogue uses c, r, v as the 3-D store maps of Q [B*Hq][T][dh] and the K / V caches
// [B*Hkv][cap][dh] (boxes of 64 x 128 x 1, encode_tmap_bf16_3d); EPI_RESIDUAL_NORM stores the
// normalised rows through v (an encode_tmap_out map like c).
struct GemmMaps {
    CUtensorMap a, b, c, r, v;
};
bool encode_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2);
cudaError_t gemm_launch(const GemmMaps& maps, const GemmArgs& args, cudaStream_t st);

// ---------------------------------------------------------------- skinny GEMM (gemm.cu)
// For a handful of activation rows (decode, M <= 64): acc[b][n] = sum_k X[b][k] W[n][k] with the
// weights as the 128-row MMA operand and the rows as the N side (padded to 16/32/64), the K range
// split over `splits` CTAs per 128 weight rows. splits == 1 with out != nullptr stores fp32 rows
// directly (out[b * ldo + n]); otherwise split s stores its partial sums in its own slice,
// ws[(s * M + b) * ldw + n], and a finalize kernel adds the slices in a fixed order (deterministic).
struct SkinnyArgs {
    int M, N, K, splits;
    float* ws;
    long long ldw;
    float* out;
    long long ldo;
    int* err;
    int w_independent;  // nonzero: the weights are not written by the previous kernel on the stream
};
constexpr int kSkinnyRowsBox = 64;  // TMA box rows of the activation operand
bool encode_skinny_x_map(CUtensorMap* map, const void* X, uint64_t rows, uint64_t K);
int skinny_splits(int N, int K);
cudaError_t gemm_skinny_launch(const CUtensorMap& tw, const CUtensorMap& tx, const SkinnyArgs& a, cudaStream_t st);

// ---------------------------------------------------------------- small kernels (kernels.cu)
cudaError_t embed_launch(const __nv_bfloat16* E, int V, int d, const int32_t* ids, int M, __nv_bfloat16* out, int* err,
                         cudaStream_t st);
cudaError_t rmsnorm_launch(const __nv_bfloat16* x, const __nv_bfloat16* g, int rows, int n, long long in_stride,
                           long long in_offset, float eps, __nv_bfloat16* y, cudaStream_t st);
cudaError_t rope_table_launch(float theta, int dh, int n_pos, __nv_bfloat16* table, cudaStream_t st);
cudaError_t pack_gate_up_launch(const __nv_bfloat16* gate, const __nv_bfloat16* up, int F, int d, __nv_bfloat16* out,
                                cudaStream_t st);
cudaError_t qknorm_rope_append_launch(const __nv_bfloat16* qkv, int B, int T, int Hq, int Hkv, int dh,
                                      const __nv_bfloat16* qg, const __nv_bfloat16* kg, const __nv_bfloat16* table,
                                      const int* len0, float eps, __nv_bfloat16* q_out, __nv_bfloat16* kc,
                                      __nv_bfloat16* vc, int cap, cudaStream_t st);
// Decode finalize kernels: sum the `splits` fp32 slices of the skinny GEMM ([splits][M][ldw]) in order,
// then apply the epilogue.
// part: [M][finalize_norm_chunks(n)] floats; tick: [M] ints, zero on entry (left zero).
int finalize_norm_chunks(int n);
cudaError_t finalize_residual_rmsnorm_launch(const float* ws, int splits, long long ldw, __nv_bfloat16* x,
                                             const __nv_bfloat16* g, int M, int n, float eps, __nv_bfloat16* y,
                                             float* part, int* tick, cudaStream_t st);
cudaError_t finalize_swiglu_launch(const float* ws, int splits, long long ldw, __nv_bfloat16* h, int M, int F,
                                   cudaStream_t st);
cudaError_t qknorm_rope_append_f32_launch(const float* ws, int splits, int B, int Hq, int Hkv, int dh, const __nv_bfloat16* qg,
                                          const __nv_bfloat16* kg, const __nv_bfloat16* table, const int* len0,
                                          float eps, __nv_bfloat16* q_out, __nv_bfloat16* kc, __nv_bfloat16* vc, int cap,
                                          const int* meta, int rolling, cudaStream_t st);
// Length bookkeeping on the device: *len = value, or *len += delta.
// Greedy next tokens of B rows of logits (row stride ld floats); see greedy_kernel. done/next/out/alive
// may be null (done null: no stop handling). work: greedy_workspace_ints(B) ints whose tickets are zero
// before the first launch (each launch leaves them zero), or null (one CTA per row).
size_t greedy_workspace_ints(int B);
cudaError_t greedy_launch(const float* logits, long long ld, int B, int V, int stop_id, int* done, int* next, int* out,
                          long long out_ld, int out_col, int* alive, int* work, cudaStream_t st);
cudaError_t copy_prefix_slots_launch(__nv_bfloat16* kc, __nv_bfloat16* vc, size_t layer_elems, int L, int nb, int Hkv,
                                     int cap, int dh, int s0, int s1, cudaStream_t st);
cudaError_t set_len_launch(int* len, int value, cudaStream_t st);
cudaError_t add_len_launch(int* len, int delta, cudaStream_t st);

// ---------------------------------------------------------------- attention (attention.cu)
// split > 0: cut each query tile's KV range into at most max_chunks chunks of >= split tiles, merged by
// the last CTA to finish; ws then holds attn_prefill_workspace() bytes whose leading ticket counters
// are zero on entry (each launch leaves them zero).
// cap: physical slots per (sequence, kv head); sm: sequence layout (SeqMap{} for plain sequences).
cudaError_t attn_prefill_launch(const __nv_bfloat16* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc, int B, int T,
                                int Hq, int Hkv, int dh, int cap, const int* len0, SeqMap sm, __nv_bfloat16* out,
                                int* err, int split, int max_chunks, float* ws, int heads, int kv_hint, cudaStream_t st);
// heads: query heads per CTA (1 or 2; 0 = chosen from the grid size). One head without a KV split runs
// the persistent kernel. kv_hint: the key count the longest query row will see (len0 + T when the host
// knows len0, else T); it only picks between two equivalent forms of the persistent kernel.
int attn_heads_per_cta(int Hq, int Hkv);
size_t attn_prefill_workspace(int B, int T, int Hq, int Hkv, int dh, int max_chunks);
void attn_prefill_split_plan(int B, int T, int Hq, int Hkv, int kv_len, int* split, int* max_chunks);
size_t attn_decode_workspace(int B, int Hq, int dh, int cap, int window, int ring);
// work: attn_decode_workspace() bytes of chunk records, merged by a second kernel; only the records of
// chunks holding keys of this call are written and read, so the workspace needs no clearing.
// err (may be null): ERR_TIMEOUT is or-ed in when a copy-ring wait gives up.
// n_keys > 0: the key count *len0 + 1 the launch will see (known on the host), which bounds the grid to
// the chunks holding keys (attn_decode_chunks of it); 0: the grid covers the whole capacity.
cudaError_t attn_decode_launch(const __nv_bfloat16* q, const __nv_bfloat16* kc, const __nv_bfloat16* vc, int B, int Hq,
                               int Hkv, int dh, int cap, const int* len0, SeqMap sm, float* work, __nv_bfloat16* out,
                               int* err, int n_keys, cudaStream_t st);
int attn_decode_chunks(int n_keys, int cap, int window, int ring);
int attn_decode_kernel_count();
// Allocation-free decode attention: size of the library's fixed scratch, and its device address on
// the current device (looked up on first use per device).
size_t attn_decode_noalloc_max_bytes();
cudaError_t attn_decode_noalloc_scratch(float** ptr);

// One-time per-process kernel attribute setup (dynamic shared memory limits); idempotent, and must
// run outside stream capture. Called by every entry point that launches these kernels.
cudaError_t gemm_prepare();
cudaError_t attention_prepare();
cudaError_t prepare_kernels();

}  // namespace q3
