/*
 * tts_decode.h — C ABI of the GB300 (sm_103a) batched decode step for
 * streaming codec-language-model text-to-speech.
 *
 * One decode step, per active stream: append this step's key/value rows to a
 * paged KV cache, attend over the stream's cache with its query rows, score
 * the result with a codebook head and pick the next codec token; in
 * speculative mode, verify K draft tokens against the target's logits.
 *
 * Sources (web pages on streaming codec-LM text-to-speech):
 *  [OPT] "Optimizing Streaming Text-to-Speech Models for Sub-50 Millisecond
 *        Latency" — "Speculative Decoding for Acoustic Tokens" (the verify
 *        rule), "Dynamic Token-Level Batching" (a static pool of 16-token KV
 *        blocks; batch membership changes at every step).
 *  [TTS] "TTS (Text-to-Speech) Serving, in depth" — "Token generation under a
 *        frame budget" (one decode step per frame, each reading the KV cache).
 *  [TON] "TontaubeV1: Streaming Text-to-Speech with Hierarchical Codec Modeling
 *        and Bounded Context" — section 3 (16,384-entry semantic and 4,096-entry
 *        acoustic codebooks plus a boundary token; later stages run at
 *        temperature zero).
 *  [NARI] "How We Made a Text-to-Speech Model Respond in Sub-50 ms" —
 *        "Additional serving optimizations" (avoid host/device synchronisation).
 *
 * Conventions shared by every call:
 *  - Every call returns a tts_status; negative values are errors.  Argument
 *    checks happen on the host before anything is launched; a call that
 *    returns an error has launched nothing.
 *  - Pointers prefixed d_ are device pointers, host_ are host pointers.  The
 *    caller allocates and owns all memory; the library keeps no pointer after
 *    a call returns.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and never synchronise the host [NARI].
 *  - Data the kernels find invalid (a block id outside the pool, a context
 *    length out of range, a draft token outside the vocabulary) never causes
 *    an out-of-bounds access: the kernel skips it, writes the defined value
 *    stated per call, and ORs a TTS_ERRBIT_* flag into *d_err (nullable,
 *    caller-owned int32 on the device; the caller reads it whenever it likes).
 *  - Tensors are dense and row-major with the shapes given per call.
 *  - Calls on different streams are thread-safe as long as their outputs and
 *    workspaces are disjoint.
 */
#ifndef TTS_DECODE_H
#define TTS_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TTS_OK = 0,
    TTS_ERR_INVALID = -1,          /* null pointer, bad size, inconsistent shape */
    TTS_ERR_UNSUPPORTED = -2,      /* a shape or type the library has no kernel for */
    TTS_ERR_WORKSPACE = -3,        /* workspace missing, misaligned or too small */
    TTS_ERR_CUDA = -4,             /* a CUDA launch or runtime call failed */
    TTS_ERR_POOL_EXHAUSTED = -5,   /* block pool has too few free blocks */
    TTS_ERR_SCRATCH_LIMIT = -6     /* request larger than the library's static scratch */
} tts_status;

enum { TTS_F32 = 0, TTS_BF16 = 1, TTS_FP8_E4M3 = 2 };  /* element types */
enum { TTS_ARGMAX = 0, TTS_GUMBEL = 1 };        /* head selection modes */
enum { TTS_VERIFY_BONUS = 1 };                  /* tts_spec_verify flags */

/* Bits ORed into *d_err by the kernels. */
enum {
    TTS_ERRBIT_BLOCK_ID = 1,   /* block table entry outside [0, num_blocks) */
    TTS_ERRBIT_CTX_LEN = 2,    /* context length outside its valid range */
    TTS_ERRBIT_TOKEN = 4,      /* draft token outside [0, V) */
    TTS_ERRBIT_TIMEOUT = 8     /* a bounded on-device wait ran out */
};

#define TTS_BLOCK_TOKENS 16

/* Paged KV cache [OPT, "Dynamic Token-Level Batching"]: a static pool of
 * num_blocks blocks of 16 tokens.  For TTS_F32 and TTS_BF16, k_pool and
 * v_pool are device arrays [num_blocks][num_kv_heads][16][head_dim] of
 * `dtype`, so each (block, head) tile is contiguous; k_scale and v_scale are
 * unused.  Supported: (TTS_BF16, head_dim 128), (TTS_F32, head_dim 64).
 *
 * TTS_FP8_E4M3 (head_dim 128; the KV cache in FP8: [OPT, "Engine-Level
 * Optimizations with TensorRT-LLM"]): every cached key or value row (one
 * token, one KV head, 128 values) is one quantisation block, stored as E4M3
 * codes with one fp32 scale, value = code * scale.  k_pool holds one
 * 4224-byte record per (block, KV head): uint8 [num_blocks][num_kv_heads][4224]
 *   bytes    0..2047  key codes: slot s, dimension d at 128 s + 16 ((d / 16)
 *                     xor (s % 8)) + d % 16 (rows of 128 bytes, 16-byte
 *                     chunks permuted as a 128-byte swizzle would)
 *   bytes 2048..4095  value codes: dimension d, slot s at 2048 + 16 d + p(s),
 *                     p(s) = 4 ((s % 8) / 2) + (s % 2) + 2 (s / 8), i.e. each
 *                     dimension's 16 slots in the order 0 1 8 9 2 3 10 11 ...
 *   bytes 4096..4159  the 16 key scales (float), 4160..4223 the value scales
 * so a tile moves with one bulk copy; v_pool is unused (NULL).  The step's
 * activations (q, k_new, v_new, the attention output) are bf16.
 * Attention on this cache runs its products in f16 on the tensor cores: the
 * queries must lie within f16's range, and every value scale below 256 (a
 * value row's largest magnitude below 114,688), else outputs are not finite.
 * Where a softmax weight times a value scale falls below 2^-22 its product
 * enters f16's subnormals: an absolute error below 2^-33 x 448 per token
 * before the division by the softmax sum.
 * All base addresses must be 16-byte aligned. */
typedef struct tts_kv_cache {
    int32_t num_blocks;
    int32_t block_size;     /* must be 16 */
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t dtype;          /* TTS_F32, TTS_BF16 or TTS_FP8_E4M3 */
    void *k_pool;
    void *v_pool;
} tts_kv_cache;

/* ------------------------------------------------------------ block pool */

/* Host-side free list of block ids [OPT, "Dynamic Token-Level Batching"]:
 * a request takes free blocks from the global pool and returns them when it
 * finishes or is aborted ("TTS Serving, in depth", "Barge-in and
 * cancellation").  Last-freed blocks are handed out first.  A pool is guarded
 * by its own mutex.  Returns TTS_ERR_INVALID for num_blocks < 1 or a null
 * `out`. */
typedef struct tts_block_pool tts_block_pool;
int tts_block_pool_create(int32_t num_blocks, tts_block_pool **out);

/* Takes n blocks, writing their ids to host_ids_out[n].  All or nothing:
 * TTS_ERR_POOL_EXHAUSTED (and no change) when fewer than n are free. */
int tts_block_pool_alloc(tts_block_pool *pool, int32_t n, int32_t *host_ids_out);

/* Returns n blocks.  All or nothing: TTS_ERR_INVALID (and no change) if any id
 * is outside the pool, not currently allocated, or repeated. */
int tts_block_pool_free(tts_block_pool *pool, const int32_t *host_ids, int32_t n);

/* Number of free blocks, or TTS_ERR_INVALID for a null pool. */
int32_t tts_block_pool_num_free(const tts_block_pool *pool);
void tts_block_pool_destroy(tts_block_pool *pool);

/* ---------------------------------------------------------------- append */

/* Writes this step's keys and values into the pool [OPT, "Dynamic Token-Level
 * Batching"]: new token j of stream b has logical position
 * s = d_ctx_before[b] + j and goes to block d_block_table[b][s / 16],
 * slot s % 16.
 *  d_block_table  int32 [B][max_blocks_per_seq]
 *  d_ctx_before   int32 [B] — tokens already cached before this step
 *  d_k_new, d_v_new  `cache->dtype` [B][q_len][num_kv_heads][head_dim]
 *                    (bf16 for a TTS_FP8_E4M3 cache)
 * FP8 cache: each new row x (head_dim values) is quantised with scale =
 * max|x| / 448 (fp32) and codes = E4M3(x / scale) (fp32 division, round to
 * nearest even, saturating at +-448); an all-zero row stores scale 0 and
 * codes 0.  The codes and the scale go to the layouts of tts_kv_cache.
 * A slot outside the table (TTS_ERRBIT_CTX_LEN) or a block id outside the
 * pool (TTS_ERRBIT_BLOCK_ID) is skipped. */
int tts_kv_append(const tts_kv_cache *cache, const int32_t *d_block_table,
                  int32_t max_blocks_per_seq, const int32_t *d_ctx_before, int32_t B,
                  int32_t q_len, const void *d_k_new, const void *d_v_new, int32_t *d_err,
                  void *stream);

/* Append with rotary position embedding fused in.  The engine of [OPT,
 * "Engine-Level Optimizations with TensorRT-LLM"] writes the KV cache and
 * applies the rotary embedding in one kernel; the rotation is RoFormer's
 * (Su et al. 2021, section 3.4) in the rotate-half arrangement.  New token j of stream b has position s = d_ctx_before[b] + j;
 * for i < 64 with angle a = s * rope_base^(-2i/128), every query and key row
 * x (128 values) becomes
 *   x[i] cos a - x[i + 64] sin a,   x[i + 64] cos a + x[i] sin a
 * (cos a and sin a from double precision, the rotation in fp32).  The query
 * rows are rewritten in place (round to nearest bf16); the rotated key rows
 * are stored as tts_kv_append stores key rows (bf16, or for an FP8 cache
 * quantised from the fp32 rotated row); value rows as tts_kv_append.
 *  d_q  bf16 [B][q_len][num_q_heads][128], in/out
 * Supported: TTS_BF16 and TTS_FP8_E4M3 caches, head_dim 128; rope_base > 1.
 * Errors as tts_kv_append; the rows of a skipped slot (TTS_ERRBIT_CTX_LEN /
 * _BLOCK_ID) are left unrotated. */
int tts_kv_append_rope(const tts_kv_cache *cache, const int32_t *d_block_table, int32_t max_blocks_per_seq,
                       const int32_t *d_ctx_before, int32_t B, int32_t q_len, int32_t num_q_heads,
                       float rope_base, void *d_q, const void *d_k_new, const void *d_v_new, int32_t *d_err,
                       void *stream);

/* ------------------------------------------------------------- attention */

/* Bytes of device workspace tts_decode_attn needs for these sizes (0 on bad
 * arguments).  Layout: scratch for the partial results of split (stream, KV
 * head) segments, then one int32 ticket per (stream, KV head) in the last
 * 256-byte-aligned part.  The workspace must be zero-filled before its first
 * use; every completed call leaves the tickets zero again (the scratch part
 * needs no particular contents), so one zeroed buffer serves any number of
 * calls on one stream.  Calls that overlap on the GPU need separate
 * workspaces. */
size_t tts_decode_attn_workspace_size(int32_t B, int32_t q_len, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim,
                                      int32_t max_ctx_len);

/* Decode attention over the paged cache [TTS, "Token generation under a frame
 * budget"; OPT, "Speculative Decoding for Acoustic Tokens" for q_len > 1]:
 * for stream b, query row j < q_len and query head h < num_q_heads,
 *   out[b][j][h] = sum_t softmax_t(scale * q[b][j][h] . k_t) v_t
 * over the stream's cached tokens t < limit, where d_ctx_lens[b] counts the
 * tokens AFTER this step's append and limit = d_ctx_lens[b] - q_len + j + 1
 * when `causal`, d_ctx_lens[b] otherwise.  Query head h reads KV head
 * h / (num_q_heads / num_kv_heads).  Runs as split-KV flash decoding with a
 * log-sum-exp merge of the splits.
 *  d_q    `cache->dtype` [B][q_len][num_q_heads][head_dim]
 *  d_out  `cache->dtype` [B][q_len][num_q_heads][head_dim]
 *  max_ctx_len  host upper bound of d_ctx_lens (sizes the grid and workspace)
 * Requires num_q_heads % num_kv_heads == 0 and
 * (num_q_heads / num_kv_heads) * q_len <= 16.  A stream whose context length
 * is outside [q_len, min(max_ctx_len, 16 * max_blocks_per_seq)] gets zeros
 * (TTS_ERRBIT_CTX_LEN); tokens in blocks with an invalid id are left out
 * (TTS_ERRBIT_BLOCK_ID). */
int tts_decode_attn(const tts_kv_cache *cache, const int32_t *d_block_table,
                    int32_t max_blocks_per_seq, const int32_t *d_ctx_lens, int32_t max_ctx_len,
                    int32_t B, int32_t q_len, int32_t num_q_heads, float scale, int32_t causal,
                    const void *d_q, void *d_out, void *d_ws, size_t ws_bytes, int32_t *d_err,
                    void *stream);

/* Decode attention with no caller workspace and no allocation.
 * The pages have no counterpart for this entry point.  It is for callers that
 * cannot call cudaMalloc where they run a decode step: engines that hand all
 * free device memory to the KV pool at start-up and so have none left to
 * allocate, plugin hosts that give a library no allocator, and real-time
 * loops that cannot absorb cudaMalloc's implicit synchronisation inside a
 * frame budget.  Same arguments and results as tts_decode_attn, without
 * d_ws / ws_bytes.  The split partials live in one 16 MiB file-scope device
 * array that every GPU loading this library holds until the process exits; a
 * request whose tts_decode_attn_workspace_size exceeds 16 MiB returns
 * TTS_ERR_SCRATCH_LIMIT and launches nothing.  The first call in a CUDA
 * context (per device, and again after that context is replaced, e.g. by
 * cudaDeviceReset) looks up the array's device address with
 * cudaGetSymbolAddress; later calls in that context reuse the address.
 * Arguments are validated before anything is queued, so a rejected call
 * leaves the array untouched.  Every call shares the one array and it keeps
 * the previous call's contents: each call clears the part that must start at
 * zero, and calls whose executions overlap on the GPU (other streams, other
 * threads) race on it.  Calls no cudaMalloc / cudaFree and no allocating
 * library routine. */
int tts_decode_attn_noalloc(const tts_kv_cache *cache, const int32_t *d_block_table,
                            int32_t max_blocks_per_seq, const int32_t *d_ctx_lens,
                            int32_t max_ctx_len, int32_t B, int32_t q_len, int32_t num_q_heads,
                            float scale, int32_t causal, const void *d_q, void *d_out,
                            int32_t *d_err, void *stream);

/* ------------------------------------------------------------------ head */

/* Bytes of device workspace tts_codebook_head_select needs (0 on bad
 * arguments).  Zero-filled before first use; left zero-filled by every call;
 * overlapping calls need separate workspaces. */
size_t tts_head_workspace_size(int32_t R, int32_t V);

/* Codebook head with fused token choice [TON, section 3]:
 *   logits[r][v] = sum_k h[r][k] * W[v][k]      (fp32 accumulation)
 * over V entries, V-1 being the boundary token.
 *  mode TTS_ARGMAX: ids[r] = argmax_v logits[r][v] (temperature zero).
 *  mode TTS_GUMBEL: ids[r] = argmax_v (logits[r][v] / temperature + G), G the
 *    Gumbel noise -log(-log u) of Philox4x64-10 uniform u with key
 *    (d_seed[r], d_step[r]) and counter (v / 8, 0, 0, 0) — a draw from
 *    softmax(logits / temperature).
 * Equal keys resolve to the lowest index.  d_eos_allowed[r] == 0 (nullable
 * array) removes v = V-1 from the choice.  The logits never leave the chip
 * unless d_logits_out is given.
 *  d_h   `dtype` [R][H];  d_W  `dtype` [V][H] (vocab-major)
 *  d_seed, d_step  uint64 [R] (read in TTS_GUMBEL mode only; may be NULL otherwise)
 *  d_ids int32 [R];  d_best float [R] (nullable: the winning key)
 *  d_logits_out float [R][V] (nullable: the speculative-verify path needs them)
 * bf16 runs on the tcgen05 tensor cores and needs H % 64 == 0 and 16-byte
 * aligned d_h, d_W; fp32 runs on CUDA cores.  Requires 1 <= R <= 4096. */
int tts_codebook_head_select(const void *d_h, const void *d_W, int32_t dtype, int32_t R,
                             int32_t H, int32_t V, int32_t mode, float temperature,
                             const uint64_t *d_seed, const uint64_t *d_step,
                             const uint8_t *d_eos_allowed, int32_t *d_ids, float *d_best,
                             float *d_logits_out, void *d_ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------- verify */

/* Speculative verification of K draft tokens per stream [OPT, "Speculative
 * Decoding for Acoustic Tokens"], for every stream b:
 *   p_t = softmax(target_logits[b][i] / temperature), p_d = draft_probs[b][i],
 *   d = draft_tokens[b][i]; draft i is accepted iff p_d[d] > 0 and
 *   u_i < p_t[d] / p_d[d], u_i the Philox uniform (key (seed[b], step[b]),
 *   counter (i / 8, 1, 0, 0)).  At the first rejection the replacement token is
 *   drawn from max(p_t - p_d, 0), normalised (Gumbel-max, counter
 *   (v / 8, 2, 0, 0); from p_t itself if that residual is zero everywhere) and
 *   verification stops.  If all K are accepted, next_token = -1, or with
 *   TTS_VERIFY_BONUS a token drawn from softmax(target_logits[b][K] /
 *   temperature) (counter (v / 8, 2, 0, 0): a stream draws at most once per
 *   call, so the draw's noise does not depend on the row drawn from).
 *  d_target_logits float [B][K+1][V];  d_draft_probs float [B][K][V]
 *  d_draft_tokens int32 [B][K];  d_seed, d_step uint64 [B]
 *  d_n_accepted, d_next_token int32 [B]
 * A draft token outside [0, V) is rejected without a draw (next_token = -1,
 * TTS_ERRBIT_TOKEN).  Requires 1 <= K <= 16 and temperature > 0. */
int tts_spec_verify(const float *d_target_logits, const float *d_draft_probs,
                    const int32_t *d_draft_tokens, int32_t B, int32_t K, int32_t V,
                    float temperature, const uint64_t *d_seed, const uint64_t *d_step,
                    int32_t flags, int32_t *d_n_accepted, int32_t *d_next_token,
                    int32_t *d_err, void *stream);

/* ------------------------------------------------------------ audio head */

/* The two-layer audio head ("TontaubeV1", section 3: each stage expands the
 * transformer state to width 4,096, applies Mish and projects to its
 * vocabulary; logits outside the stage's target vocabulary are masked at
 * sampling), batched over R rows:
 *   z[r][f] = bfloat16(Mish(sum_k h[r][k] W1[f][k] + b1[f])),
 *             Mish(x) = x tanh(ln(1 + e^x)), computed in fp32;
 *   logit[r][v] = fp32(sum_f z[r][f] W2[v][f] + b2[v]);
 * then the choice of tts_codebook_head_select over the ids row r may take:
 * every id below V - n_tail, and id V - n_tail + j when bit j of
 * d_tail_allowed[r] is set (the stage's structural tokens; NULL: all
 * allowed).  E.g. CB0: V = 16386 with n_tail = 2 (row terminator,
 * <|audio_split|>); an acoustic stage: V = 4097, n_tail = 1 (the boundary).
 *  d_h bf16 [R][H];  d_W1 bf16 [F][H];  d_b1 float [F] or NULL;
 *  d_W2 bf16 [V][F];  d_b2 float [V] or NULL;  d_tail_allowed uint32 [R];
 *  d_z bf16 [R][F], written (caller-owned, 16-byte aligned);
 *  d_ids, d_best, d_logits_out, d_seed, d_step, mode, temperature, d_ws and
 *  ws_bytes as tts_codebook_head_select (workspace tts_head_workspace_size(R, V)).
 * Requires H and F multiples of 64, 0 <= n_tail <= 32.  Two kernels on
 * `stream`; the projection starts streaming W2 while the first layer finishes.
 * TTS_ERR_UNSUPPORTED for other shapes; TTS_ERR_INVALID for bad pointers or
 * arguments. */
int tts_audio_head_select(const void *d_h, const void *d_W1, const float *d_b1, const void *d_W2,
                          const float *d_b2, int32_t R, int32_t H, int32_t F, int32_t V, int32_t n_tail,
                          const uint32_t *d_tail_allowed, int32_t mode, float temperature,
                          const uint64_t *d_seed, const uint64_t *d_step, void *d_z, int32_t *d_ids,
                          float *d_best, float *d_logits_out, void *d_ws, size_t ws_bytes, void *stream);

/* ----------------------------------------------------------- full step */

/* One decode step in one call: tts_kv_append (tts_kv_append_rope when
 * rope_base != 0: d_q is then rotated in place, so a repeated call on the same
 * d_q rotates it again), then tts_decode_attn into d_attn_out, then
 * tts_codebook_head_select with h = d_attn_out read as
 * [B * q_len][num_q_heads * head_dim] (dtype cache->dtype; bf16 for an FP8
 * cache; R = B * q_len).
 * Arguments mean what they mean for those calls; all of them are
 * checked before anything is launched.  The attention and head kernels are
 * launched as programmatic dependents of the kernel before them: each starts
 * its set-up (tile map; weight stream) while its predecessor finishes, and
 * waits for it before reading the KV pool or the attention output.  So the
 * caller must not write the step's inputs (q, k_new, v_new, tables, lengths,
 * weights, seeds) from the kernels of this same call — only before it. */
int tts_decode_step(const tts_kv_cache *cache, const int32_t *d_block_table,
                    int32_t max_blocks_per_seq, const int32_t *d_ctx_before,
                    const int32_t *d_ctx_lens, int32_t max_ctx_len, int32_t B, int32_t q_len,
                    int32_t num_q_heads, float scale, int32_t causal, float rope_base, void *d_q,
                    const void *d_k_new, const void *d_v_new, void *d_attn_out, void *d_attn_ws,
                    size_t attn_ws_bytes, const void *d_W, int32_t V, int32_t mode,
                    float temperature, const uint64_t *d_seed, const uint64_t *d_step,
                    const uint8_t *d_eos_allowed, int32_t *d_ids, float *d_best,
                    float *d_logits_out, void *d_head_ws, size_t head_ws_bytes, int32_t *d_err,
                    void *stream);

/* ------------------------------------------------------- captured step */

/* A decode step captured once as a CUDA graph for fixed shapes and fixed
 * buffers ("How We Made a TTS Model Respond in Sub-50 ms", section
 * "Additional serving optimizations": graphs captured for a predefined set of
 * batch sizes; "Optimizing Streaming Text-to-Speech Models for Sub-50
 * Millisecond Latency", section "Engine-Level Optimizations with
 * TensorRT-LLM": the CPU only starts the graph).  No counterpart API on the
 * pages.  Each launch:
 *   1. copies input_bytes from h_inputs (pinned host memory) to d_inputs with
 *      a kernel reading the host buffer through unified addressing;
 *   2. runs tts_decode_step with the fields below (the step's input pointers
 *      normally point into d_inputs, so step 1 refreshes them);
 *   3. writes d_ids[0..R) to h_ids (pinned host memory, R = B * q_len) and,
 *      if h_boundary_count is not NULL, the number of rows whose id is the
 *      boundary token V - 1 to *h_boundary_count (a device-side end-of-stream
 *      flag: the host tests one word instead of scanning the ids).
 * The caller writes a step's inputs into h_inputs, launches, synchronises the
 * stream (or an event after the launch), and reads h_ids.  Every buffer is
 * owned by the caller and must outlive the graph; the descriptor is read only
 * by tts_step_graph_create.  Fields mean what tts_decode_step's arguments
 * mean. */
typedef struct {
    const tts_kv_cache *cache;
    const int32_t *d_block_table;
    int32_t max_blocks_per_seq;
    const int32_t *d_ctx_before;
    const int32_t *d_ctx_lens;
    int32_t max_ctx_len;
    int32_t B;
    int32_t q_len;
    int32_t num_q_heads;
    float scale;
    int32_t causal;
    float rope_base;
    void *d_q;
    const void *d_k_new;
    const void *d_v_new;
    void *d_attn_out;
    void *d_attn_ws;
    size_t attn_ws_bytes;
    const void *d_W;
    int32_t V;
    int32_t mode;
    float temperature;
    const uint64_t *d_seed;
    const uint64_t *d_step;
    const uint8_t *d_eos_allowed;
    int32_t *d_ids;
    float *d_best;
    float *d_logits_out;
    void *d_head_ws;
    size_t head_ws_bytes;
    int32_t *d_err;
    const void *h_inputs;       /* pinned host, 16-byte aligned */
    void *d_inputs;             /* device, 16-byte aligned */
    size_t input_bytes;         /* multiple of 16 */
    int32_t *h_ids;             /* pinned host [R] */
    int32_t *h_boundary_count;  /* pinned host, nullable */
    /* Optional verify stage (when d_n_accepted is not NULL): the captured
     * step ends with tts_spec_verify over the head's logits (d_logits_out,
     * [B][q_len][V] with q_len = K + 1), and the accepted counts and next
     * tokens are also written to h_n_accepted / h_next_token (pinned host,
     * nullable).  Fields mean what tts_spec_verify's arguments mean. */
    const float *d_draft_probs;     /* [B][K][V] */
    const int32_t *d_draft_tokens;  /* [B][K] */
    float verify_temperature;
    int32_t verify_flags;
    const uint64_t *d_vseed;        /* [B] */
    const uint64_t *d_vstep;        /* [B] */
    int32_t *d_n_accepted;          /* [B] */
    int32_t *d_next_token;          /* [B] */
    int32_t *h_n_accepted;          /* pinned host [B], nullable */
    int32_t *h_next_token;          /* pinned host [B], nullable */
} tts_step_graph_desc;

typedef struct tts_step_graph tts_step_graph;

/* Checks every field (TTS_ERR_INVALID / _UNSUPPORTED / _WORKSPACE as
 * tts_decode_step; TTS_ERR_INVALID for host buffers that are not pinned or
 * misaligned transfer buffers), captures and instantiates the graph.  On
 * success *out owns it.  Does not launch anything; the attention and head
 * workspaces must be zero-filled before the first launch. */
int tts_step_graph_create(const tts_step_graph_desc *desc, tts_step_graph **out);

/* Launches the captured step on `stream` (asynchronous). */
int tts_step_graph_launch(tts_step_graph *graph, void *stream);

/* Launches the captured step on `stream` and returns once its ids (and the
 * boundary count) are in the pinned host buffers: a serving loop's call.  For
 * a bf16 / FP8 step without a verify stage, the head's last CTA writes a
 * launch number to pinned host memory after the ids (system-scope fence
 * between), and this call spins on that number instead of synchronising the
 * stream (at most a second, then it synchronises the stream, which also
 * reports a failed launch); the launch's last CTAs may still be exiting when
 * it returns (later work on the stream is ordered after them as usual).
 * Other steps: launch, then cudaStreamSynchronize.  TTS_ERR_CUDA on a launch
 * or stream error. */
int tts_step_graph_run(tts_step_graph *graph, void *stream);

/* Frees the graph (no GPU work of it may still be pending).  NULL is a no-op. */
void tts_step_graph_destroy(tts_step_graph *graph);

/* Captured steps for a set of batch sizes ("How We Made a TTS Model Respond
 * in Sub-50 ms", section "Additional serving optimizations": graphs are
 * captured for a predefined set of batch sizes, and an oversize cohort is
 * split rather than run eagerly).  `desc` describes the step for the largest
 * size (desc->B); every per-stream array it points to (and h_inputs /
 * d_inputs) is laid out for desc->B streams.  The packed inputs consist of
 * n_segs regions: region i starts at byte seg_offset[i] (a multiple of 16) of
 * h_inputs and d_inputs and holds seg_row_bytes[i] bytes (a multiple of 4) per
 * stream, streams in order.  For each size b in sizes[] (strictly increasing,
 * the last equal to desc->B, at most TTS_GRAPH_SET_MAX of them) one graph is
 * captured that runs the step on the first b streams: it copies the first b
 * rows of every region, runs tts_decode_step with B = b on the same buffers,
 * and writes b * q_len ids (and their boundary count) to h_ids.
 * Errors as tts_step_graph_create; TTS_ERR_INVALID for bad sizes or regions
 * outside input_bytes. */
#define TTS_GRAPH_SET_MAX 16
typedef struct tts_step_graph_set tts_step_graph_set;
int tts_step_graph_set_create(const tts_step_graph_desc *desc, const int32_t *sizes, int32_t n_sizes,
                              const size_t *seg_offset, const size_t *seg_row_bytes, int32_t n_segs,
                              tts_step_graph_set **out);

/* Launches the graph of the smallest captured size b >= n_streams (its size
 * in *chosen_B if not NULL).  The caller has written the inputs of streams
 * 0..n_streams-1 and made streams n_streams..b-1 harmless (e.g. a table row
 * holding a scratch block, ctx_before 0); their ids are to be ignored.
 * TTS_ERR_INVALID if n_streams exceeds the largest size (split the cohort). */
int tts_step_graph_set_launch(tts_step_graph_set *set, int32_t n_streams, int32_t *chosen_B, void *stream);

/* tts_step_graph_set_launch, then the wait of tts_step_graph_run: returns
 * once the launch's ids are in the pinned host buffers (one launch number is
 * shared by every size of the set, so launch a set on one stream at a time). */
int tts_step_graph_set_run(tts_step_graph_set *set, int32_t n_streams, int32_t *chosen_B, void *stream);

/* Frees every graph of the set (no GPU work of it may still be pending). */
void tts_step_graph_set_destroy(tts_step_graph_set *set);

/* ------------------------------------------------------ code predictor */

/* The code predictor's frame loop ("How We Made a TTS Model Respond in
 * Sub-50 ms", sections "Exploiting the regular building of the Code
 * Predictor" and "Turn a fixed predictor loop into one GPU program": a fixed
 * number of autoregressive steps per frame, one per remaining codebook, over
 * a short bounded context in a preallocated KV cache).  For every stream r,
 * with x = x0[r] and an empty cache, step i = 0 .. n_steps-1 computes
 *   q, k, v = bf16(x Wqkv^T)      (q: the first Hq*D features, then k, v)
 *   k, v appended at position i of the stream's cache
 *   o = bf16(attention of q over positions 0..i), scale 1/sqrt(head_dim),
 *       query head h reading KV head h / (Hq/Hkv)
 *   tokens[i][r] = argmax_v (o . W_i[v]), or with TTS_GUMBEL the argmax of
 *       logit / T + Gumbel noise (Philox key (seed[r], step[r]), counter
 *       (v / 8, 0, i + 1, 0), half v % 8)
 *   x = E_i[tokens[i][r]]
 * Fields: R streams; H = num_q_heads * head_dim (the width of x and of o);
 * head_dim 128; n_steps <= 16 (one 16-token block per stream);
 *  d_x0 bf16 [R][H];  d_Wqkv bf16 [(Hq + 2 Hkv) * head_dim][H];
 *  d_W bf16 [n_steps][V][H];  d_E bf16 [n_steps][V][H];
 *  d_tokens int32 [n_steps][R] (written);  d_seed, d_step uint64 [R] (Gumbel);
 *  d_ws: workspace of tts_code_predictor_workspace_size bytes, 256-byte
 *  aligned, caller-owned; it holds x, q, k, v, o, the cache and the kernels'
 *  workspaces (any contents on entry).  d_err as tts_decode_step. */
typedef struct {
    int32_t R;
    int32_t H;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t V;
    int32_t n_steps;
    int32_t mode;
    float temperature;
    const void *d_x0;
    const void *d_Wqkv;
    const void *d_W;
    const void *d_E;
    const uint64_t *d_seed;
    const uint64_t *d_step;
    int32_t *d_tokens;
    void *d_ws;
    size_t ws_bytes;
    int32_t *d_err;
    int32_t flags;  /* TTS_PREDICTOR_MULTI_KERNEL: one kernel per stage, not one launch */
} tts_code_predictor_desc;

/* By default the frame runs as one cooperative persistent kernel (one CTA
 * per SM, three grid barriers per step) when R <= 64, H <= 1024, head_dim is
 * 128 and (Hq + 2 Hkv) * 128 and V are multiples of 16; otherwise, or with
 * this flag, as 4-5 kernels per step. */
#define TTS_PREDICTOR_MULTI_KERNEL 1

/* Workspace bytes for the loop (0 for unsupported sizes). */
size_t tts_code_predictor_workspace_size(int32_t R, int32_t H, int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t V, int32_t n_steps);

/* Runs one frame's loop on `stream` (the persistent kernel, or 4-5 kernels
 * per step, each a programmatic dependent of the one before).  TTS_ERR_INVALID /
 * _UNSUPPORTED / _WORKSPACE as the step's calls. */
int tts_code_predictor_run(const tts_code_predictor_desc *desc, void *stream);

/* The same loop captured once as a CUDA graph for the descriptor's buffers
 * (the caller writes x0, seeds and steps before each launch; the workspace
 * and outputs must outlive the graph). */
typedef struct tts_code_predictor_graph tts_code_predictor_graph;
int tts_code_predictor_graph_create(const tts_code_predictor_desc *desc, tts_code_predictor_graph **out);
int tts_code_predictor_graph_launch(tts_code_predictor_graph *graph, void *stream);
void tts_code_predictor_graph_destroy(tts_code_predictor_graph *graph);

/* ------------------------------------------------------ launch options */

/* No counterpart on the pages: kernel-launch plumbing.  With
 * TTS_LAUNCH_PROGRAMMATIC set, the single-kernel calls this thread makes
 * afterwards (tts_kv_append, tts_kv_append_rope, tts_decode_attn,
 * tts_codebook_head_select) launch their kernel as a
 * programmatic dependent of the previous kernel in the stream: it may start
 * while that kernel finishes (hiding the launch latency, as the kernels of
 * tts_decode_step do) and waits for its completion before touching anything
 * that kernel may write, except: tts_decode_attn reads d_ctx_lens and
 * d_block_table, and tts_codebook_head_select reads d_W, before that wait,
 * so the previous kernel must not write those.  The setting is per calling
 * thread.  Returns the previous flags. */
enum { TTS_LAUNCH_PROGRAMMATIC = 1 };
int32_t tts_set_launch_flags(int32_t flags);

/* Test support (no counterpart on the pages): makes a bounded on-device wait
 * run out, to test the timeout path without faulting or hanging a GPU.  For
 * the calls this thread makes afterwards, every wait of the kernels below
 * gives up after wait_limit_cycles SM clock cycles (default 2e9, about one
 * second) and, with
 *   TTS_TEST_STALL_ATTN_RING: each warp of tts_decode_attn's bf16 / FP8
 *     kernel expects 16 more bytes on its first ring stage than its copies
 *     deliver, so its first wait runs out;
 *   TTS_TEST_STALL_PREDICTOR_GRID: the persistent code-predictor kernel's
 *     first grid barrier waits for one CTA more than the grid has.
 * The kernel then ORs TTS_ERRBIT_TIMEOUT into *d_err, stops issuing work,
 * waits (bounded) for the copies it issued, and returns; its outputs are
 * undefined.  TTS_TEST_STALL_NONE restores normal operation.
 * TTS_ERR_INVALID for an unknown mode or a limit outside [1e3, 4e9]. */
enum { TTS_TEST_STALL_NONE = 0, TTS_TEST_STALL_ATTN_RING = 1, TTS_TEST_STALL_PREDICTOR_GRID = 2 };
int tts_test_set_stall(int32_t what, int64_t wait_limit_cycles);

/* Test support (no counterpart on the pages): the Gumbel noise every Gumbel
 * draw of the library uses (head, verify, code predictor), -ln(-ln u), for n
 * 32-bit Philox words:
 * u = (2 (bits >> 9) + 1) / 2^24, so that a test can bound its distance to
 * the exact value over every u.  d_bits uint32 [n], d_out float [n] (device);
 * enqueued on `stream`.  TTS_ERR_INVALID for n < 0 or a null pointer with
 * n > 0. */
int tts_test_gumbel_noise(const uint32_t *d_bits, float *d_out, int32_t n, void *stream);

/* ----------------------------------------------------------------- misc */

/* Static description of a status code. */
const char *tts_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int tts_version(void);

#ifdef __cplusplus
}
#endif
#endif /* TTS_DECODE_H */
