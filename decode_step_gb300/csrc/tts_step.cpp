// tts_decode_step: one decode step (append, attention, head) in one call.
//
// Every argument of the three stages is checked before anything is launched.
// The attention kernel and the head are launched as programmatic dependents
// of the kernel before them, so each one's set-up (the attention's tile map,
// the head's weight stream) overlaps the tail of its predecessor; both wait
// (griddepcontrol.wait) before reading what the predecessor writes (the KV
// pool; the attention output).
#include <cuda_runtime.h>

#include "tts_decode.h"
#include "tts_internal.h"

extern "C" int tts_decode_step(const tts_kv_cache *cache, const int32_t *d_block_table,
                               int32_t max_blocks_per_seq, const int32_t *d_ctx_before,
                               const int32_t *d_ctx_lens, int32_t max_ctx_len, int32_t B,
                               int32_t q_len, int32_t num_q_heads, float scale, int32_t causal,
                               float rope_base, void *d_q, const void *d_k_new, const void *d_v_new,
                               void *d_attn_out, void *d_attn_ws, size_t attn_ws_bytes,
                               const void *d_W, int32_t V, int32_t mode, float temperature,
                               const uint64_t *d_seed, const uint64_t *d_step,
                               const uint8_t *d_eos_allowed, int32_t *d_ids, float *d_best,
                               float *d_logits_out, void *d_head_ws, size_t head_ws_bytes,
                               int32_t *d_err, void *stream) {
    using namespace tts;
    if (!cache) return TTS_ERR_INVALID;
    if (B == 0) return TTS_OK;
    AppendLaunch ap;
    AttnLaunch at;
    HeadLaunch hd;
    int st = prepare_append_rope(cache, d_block_table, max_blocks_per_seq, d_ctx_before, B, q_len, num_q_heads,
                                 rope_base, d_q, d_k_new, d_v_new, d_err, &ap);
    if (st != TTS_OK) return st;
    st = prepare_attn(cache, d_block_table, max_blocks_per_seq, d_ctx_lens, max_ctx_len, B, q_len,
                      num_q_heads, scale, causal, d_q, d_attn_out, d_attn_ws, attn_ws_bytes, d_err, &at);
    if (st != TTS_OK) return st;
    const long long R = static_cast<long long>(B) * q_len;
    const long long H = static_cast<long long>(num_q_heads) * cache->head_dim;
    if (R > 0x7FFFFFFF || H > 0x7FFFFFFF) return TTS_ERR_INVALID;
    st = prepare_head(d_attn_out, d_W, cache->dtype == TTS_FP8_E4M3 ? TTS_BF16 : cache->dtype, static_cast<int32_t>(R), static_cast<int32_t>(H), V,
                      mode, temperature, d_seed, d_step, d_eos_allowed, d_ids, d_best, d_logits_out,
                      d_head_ws, head_ws_bytes, &hd);
    if (st != TTS_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = launch_append(ap, {s, false});
    if (st != TTS_OK) return st;
    st = launch_attn(at, {s, true});
    if (st != TTS_OK) return st;
    return launch_head(hd, {s, true});
}
