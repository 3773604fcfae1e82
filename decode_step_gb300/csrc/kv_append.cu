// KV append: scatter this step's key/value rows into the paged pool
// ("Optimizing Streaming Text-to-Speech Models for Sub-50 Millisecond
// Latency", section "Dynamic Token-Level Batching": a static pool of 16-token
// blocks; token s of a stream lives in block table[s / 16], slot s % 16).
//
// One CTA per (stream, new token); its threads copy the token's Hkv rows of K
// and of V as 16-byte vectors.  Pure data movement: bytes per launch =
// 2 (read + write) x 2 (K, V) x B x q_len x Hkv x row bytes.
#include "tts_common.cuh"
#include "tts_internal.h"

namespace tts {
namespace {

__global__ void __launch_bounds__(128)
kv_append_kernel(const int32_t *__restrict__ table, int max_blocks,
                 const int32_t *__restrict__ ctx_before, int q_len, int Hkv, int num_blocks,
                 int row_vecs, const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                 uint4 *__restrict__ k_pool, uint4 *__restrict__ v_pool, int32_t *err) {
    pdl_wait_prerequisites();
    pdl_allow_dependents();
    const int b = blockIdx.x / q_len;
    const int j = blockIdx.x % q_len;
    const int before = ctx_before[b];
    const int cap = max_blocks * TTS_BLOCK_TOKENS;
    if (before < 0 || before >= cap || j >= cap - before) {
        if (threadIdx.x == 0) flag_error(err, TTS_ERRBIT_CTX_LEN);
        return;
    }
    const int s = before + j;
    const int blk = table[static_cast<size_t>(b) * max_blocks + s / TTS_BLOCK_TOKENS];
    if (blk < 0 || blk >= num_blocks) {
        if (threadIdx.x == 0) flag_error(err, TTS_ERRBIT_BLOCK_ID);
        return;
    }
    const int slot = s % TTS_BLOCK_TOKENS;
    const int per_tensor = Hkv * row_vecs;
    const size_t src0 = static_cast<size_t>(blockIdx.x) * per_tensor;
    for (int i = threadIdx.x; i < 2 * per_tensor; i += blockDim.x) {
        const bool is_v = i >= per_tensor;
        const int e = is_v ? i - per_tensor : i;
        const int g = e / row_vecs;
        const int c = e % row_vecs;
        const size_t dst =
            ((static_cast<size_t>(blk) * Hkv + g) * TTS_BLOCK_TOKENS + slot) * row_vecs + c;
        if (is_v)
            v_pool[dst] = __ldg(v_new + src0 + e);
        else
            k_pool[dst] = __ldg(k_new + src0 + e);
    }
}

}  // namespace
}  // namespace tts

namespace tts {

int prepare_append(const tts_kv_cache *cache, const int32_t *d_block_table, int32_t max_blocks_per_seq,
                   const int32_t *d_ctx_before, int32_t B, int32_t q_len, const void *d_k_new,
                   const void *d_v_new, int32_t *d_err, AppendLaunch *out) {
    if (!cache || !d_block_table || !d_ctx_before || !d_k_new || !d_v_new) return TTS_ERR_INVALID;
    if (!cache->k_pool || !cache->v_pool) return TTS_ERR_INVALID;
    if (B < 0 || q_len < 1 || max_blocks_per_seq < 1 || max_blocks_per_seq > (1 << 20) ||
        cache->num_blocks < 1 || cache->num_kv_heads < 1 || cache->head_dim < 1)
        return TTS_ERR_INVALID;
    if (cache->block_size != TTS_BLOCK_TOKENS) return TTS_ERR_UNSUPPORTED;
    if (cache->dtype != TTS_F32 && cache->dtype != TTS_BF16) return TTS_ERR_UNSUPPORTED;
    const int elem = cache->dtype == TTS_F32 ? 4 : 2;
    const long row_bytes = static_cast<long>(cache->head_dim) * elem;
    if (row_bytes % 16 != 0) return TTS_ERR_UNSUPPORTED;
    if (!aligned16(cache->k_pool) || !aligned16(cache->v_pool) || !aligned16(d_k_new) ||
        !aligned16(d_v_new))
        return TTS_ERR_INVALID;
    if (static_cast<long>(B) * q_len > 0x7FFFFFFFL) return TTS_ERR_INVALID;
    *out = AppendLaunch{cache, d_block_table, max_blocks_per_seq, d_ctx_before, B, q_len, d_k_new, d_v_new, d_err};
    return TTS_OK;
}

int launch_append(const AppendLaunch &L, LaunchOpts o) {
    if (L.B == 0) return TTS_OK;
    const int elem = L.cache->dtype == TTS_F32 ? 4 : 2;
    const int row_vecs = L.cache->head_dim * elem / 16;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(static_cast<long>(L.B) * L.q_len), 1, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.stream = o.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = o.pdl ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kv_append_kernel, L.table, L.max_blocks, L.ctx_before, L.q_len,
                           static_cast<int>(L.cache->num_kv_heads), static_cast<int>(L.cache->num_blocks),
                           row_vecs, static_cast<const uint4 *>(L.k_new), static_cast<const uint4 *>(L.v_new),
                           static_cast<uint4 *>(L.cache->k_pool), static_cast<uint4 *>(L.cache->v_pool),
                           L.err) != cudaSuccess) {
        cudaGetLastError();
        return TTS_ERR_CUDA;
    }
    return TTS_OK;
}

}  // namespace tts

extern "C" int tts_kv_append(const tts_kv_cache *cache, const int32_t *d_block_table,
                             int32_t max_blocks_per_seq, const int32_t *d_ctx_before, int32_t B,
                             int32_t q_len, const void *d_k_new, const void *d_v_new,
                             int32_t *d_err, void *stream) {
    tts::AppendLaunch L;
    const int st = tts::prepare_append(cache, d_block_table, max_blocks_per_seq, d_ctx_before, B, q_len,
                                       d_k_new, d_v_new, d_err, &L);
    if (st != TTS_OK) return st;
    return tts::launch_append(L, {static_cast<cudaStream_t>(stream), false});
}
